// drivers.cuh -- the scan kernels: env-major (general and one-tile fast),
// time-major (general, fast, and staged through a shared-memory ring).  See
// scan_core.cuh for the scan structure they share and estimators.cuh for the
// estimator interface.
#pragma once

#include "estimators.cuh"
#include "tma.cuh"

namespace rlca {

// ---------------------------------------------------------------------------
// env-major driver
// ---------------------------------------------------------------------------
template <class Est, int TPR>
__global__ void __launch_bounds__(EmShape<TPR>::BLOCK)
    em_scan_kernel(Est est, Geom g) {
  using S = EmShape<TPR>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  constexpr int L = S::L, GW = S::GW, NWR = S::NWR;

  extern __shared__ __align__(16) unsigned char smem[];
  Aff<V>* xw = reinterpret_cast<Aff<V>*>(smem);  // [2][ROWS][NWR] warp totals (NWR > 1)
  unsigned char* est_smem = smem + (NWR > 1 ? 2 * S::ROWS * NWR * sizeof(Aff<V>) : 0);

  const int tid = threadIdx.x;
  const int j = tid % TPR;
  const int rloc = tid / TPR;
  const int lane = tid & 31;
  const int lig = j % GW;
  const int wr = j / 32;
  const int seg = g.nseg == 1 ? 0 : (int)(blockIdx.x % (unsigned)g.nseg);
  const int64_t row0 = (int64_t)(g.nseg == 1 ? blockIdx.x : blockIdx.x / (unsigned)g.nseg) * S::ROWS;
  const int64_t row = row0 + rloc;
  const bool row_ok = row < g.E;
  const int seg_lo = seg * g.seg_len;
  const int seg_hi = min(g.T, seg_lo + g.seg_len);
  const bool vec = g.vec != 0;
  const bool agg_mode = g.mode == kModeAggregate;
  const EnvMajor lay{g.E, g.T};
  const bool early = g.early != 0 && g.nseg == 1 && !agg_mode;
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (!early) pdl_wait();

  Aff<V> carry;
  if (agg_mode) {
    carry = aff_identity<V>();
  } else {
    V c0 = row_ok ? est.row_carry(row) : V(0);
    if (g.nseg > 1 && row_ok) c0 = segment_carry_in<V, BWD>(g, row, seg, c0);
    carry = {c0, V(0)};
  }

  const int ntiles = (seg_hi - seg_lo + S::TILE - 1) / S::TILE;
  for (int it = 0; it < ntiles; ++it) {
    const int tile = BWD ? ntiles - 1 - it : it;
    const int ts = seg_lo + tile * S::TILE;
    const int te = min(seg_hi, ts + S::TILE);
    const int t0 = ts + j * L;
    const int n = row_ok ? max(0, min(L, te - t0)) : 0;

    est.template stage<S::ROWS, S::BLOCK, S::TILE>(lay, g, row0, rloc, ts, te, est_smem);
    typename Est::template Regs<L> R;
    const GIO<EnvMajor, false, typename Est::Store> io{lay, row, t0, n, vec};
    est.template load<L>(R, io, rloc, ts, S::TILE, S::ROWS, est_smem);

    if constexpr (Est::kNb > 0) {
      // neighbour step's inputs: from the adjacent lane when it holds them,
      // else straight from memory
      float give[Est::kNb > 0 ? Est::kNb : 1], got[Est::kNb > 0 ? Est::kNb : 1];
      est.nb_give(R, give);
#pragma unroll
      for (int i = 0; i < Est::kNb; ++i)
        got[i] = BWD ? __shfl_down_sync(kFullMask, give[i], 1, GW) : __shfl_up_sync(kFullMask, give[i], 1, GW);
      const int tn = BWD ? t0 + L : t0 - 1;
      const bool edge = BWD ? (lig == GW - 1 || t0 + L >= te) : (lig == 0);
      if (n > 0 && edge && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T))
        est.nb_load(lay, row, tn, got);
      est.nb_take(R, got);
    }

    Aff<V> c[L];
#pragma unroll
    for (int k = 0; k < L; ++k) c[k] = (k < n) ? est.coef(R, k, t0 + k) : aff_identity<V>();
    Aff<V> agg = aff_identity<V>();
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) agg = compose(c[k], agg);
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) agg = compose(c[k], agg);
    }

    // inclusive scan of the thread maps inside the row's lane group
    Aff<V> inc = agg;
#pragma unroll
    for (int off = 1; off < GW; off <<= 1) {
      if (BWD) {
        Aff<V> o = shfl_down_aff(inc, off, GW);
        if (lig + off < GW) inc = compose(inc, o);
      } else {
        Aff<V> o = shfl_up_aff(inc, off, GW);
        if (lig >= off) inc = compose(inc, o);
      }
    }
    Aff<V> exc = BWD ? shfl_down_aff(inc, 1, GW) : shfl_up_aff(inc, 1, GW);
    if (lig == (BWD ? GW - 1 : 0)) exc = aff_identity<V>();

    Aff<V> boundary, next_carry;
    if constexpr (NWR > 1) {
      // warp totals of the row through shared memory, then every warp scans
      // the NWR totals with shuffles (lanes >= NWR hold the identity)
      Aff<V>* x = xw + ((it & 1) * S::ROWS + rloc) * NWR;
      if (lane == (BWD ? 0 : 31)) x[wr] = inc;
      __syncthreads();
      Aff<V> tw = lane < NWR ? x[lane] : aff_identity<V>();
#pragma unroll
      for (int off = 1; off < NWR; off <<= 1) {
        if (BWD) {
          Aff<V> o = shfl_down_aff(tw, off, 32);
          if (lane + off < NWR) tw = compose(tw, o);
        } else {
          Aff<V> o = shfl_up_aff(tw, off, 32);
          if (lane >= off) tw = compose(tw, o);
        }
      }
      // maps of the warps after (backward) / before (forward) this one
      const int src = BWD ? wr + 1 : wr - 1;
      Aff<V> ex = shfl_idx_aff(tw, src & 31, 32);
      if (BWD ? (wr == NWR - 1) : (wr == 0)) ex = aff_identity<V>();
      boundary = compose(ex, carry);
      next_carry = compose(shfl_idx_aff(tw, BWD ? 0 : NWR - 1, 32), carry);
    } else {
      boundary = carry;
      Aff<V> tot = shfl_idx_aff(inc, BWD ? 0 : GW - 1, GW);
      next_carry = compose(tot, carry);
    }

    if (!agg_mode) {
      V A = compose(exc, boundary).a;  // value just outside this thread's chunk
      if (BWD) {
#pragma unroll
        for (int k = L - 1; k >= 0; --k) {
          V adj = A;
          A = c[k].a + c[k].b * A;
          est.emit(R, k, A, adj, c[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < L; ++k) {
          V adj = A;
          A = c[k].a + c[k].b * A;
          est.emit(R, k, A, adj, c[k]);
        }
      }
      if (early && it == 0) pdl_wait();  // the previous kernel may still read or write what we overwrite
      est.template store<L>(R, io);
    }
    carry = next_carry;
  }
  if (agg_mode && row_ok && j == 0 && in_range(row * g.nseg + seg, g.E * (int64_t)g.nseg))
    reinterpret_cast<Aff<V>*>(g.ws)[row * g.nseg + seg] = carry;
}

// ---------------------------------------------------------------------------
// the fast env-major driver's scan of one row group whose inputs are in R:
// neighbour exchange, coefficients, warp scan, cross-warp exchange through
// xw ([ROWS][NWR] slots, one CTA barrier), re-expansion into R's outputs.
// Every thread of the CTA calls it (the barrier).
// ---------------------------------------------------------------------------
template <class Est, int TPR, int LS>
__device__ __forceinline__ void em_fast_scan(const Est& est, typename Est::template Regs<EmShape<TPR, LS>::L>& R,
                                             const Geom& g, const EnvMajor& lay, int64_t row, int t0, bool active,
                                             int rloc, Aff<typename Est::V>* xw) {
  using S = EmShape<TPR, LS>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  constexpr int L = S::L, GW = S::GW, NWR = S::NWR;
  const int j = threadIdx.x % TPR;
  const int lane = threadIdx.x & 31;
  const int lig = j % GW;
  const int wr = j / 32;
  if constexpr (Est::kNb > 0) {
    float give[Est::kNb > 0 ? Est::kNb : 1], got[Est::kNb > 0 ? Est::kNb : 1];
    est.nb_give(R, give);
#pragma unroll
    for (int i = 0; i < Est::kNb; ++i)
      got[i] = BWD ? __shfl_down_sync(kFullMask, give[i], 1, GW) : __shfl_up_sync(kFullMask, give[i], 1, GW);
    // a row fits in one tile: the neighbour lies in the same row group except
    // across warps of a long row
    if constexpr (NWR > 1) {
      const int tn = BWD ? t0 + L : t0 - 1;
      const bool edge = BWD ? (lane == 31) : (lane == 0);
      if (active && edge && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T))
        est.nb_load(lay, row, tn, got);
    }
    est.nb_take(R, got);
  }

  Aff<V> c[L];
#pragma unroll
  for (int k = 0; k < L; ++k) c[k] = est.coef(R, k, t0 + k);
  Aff<V> agg = aff_identity<V>();
  if (BWD) {
#pragma unroll
    for (int k = L - 1; k >= 0; --k) agg = compose(c[k], agg);
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) agg = compose(c[k], agg);
  }
  if (!active) agg = aff_identity<V>();

  Aff<V> inc = agg;
#pragma unroll
  for (int off = 1; off < GW; off <<= 1) {
    if (BWD) {
      Aff<V> o = shfl_down_aff(inc, off, GW);
      if (lig + off < GW) inc = compose(inc, o);
    } else {
      Aff<V> o = shfl_up_aff(inc, off, GW);
      if (lig >= off) inc = compose(inc, o);
    }
  }
  Aff<V> exc = BWD ? shfl_down_aff(inc, 1, GW) : shfl_up_aff(inc, 1, GW);
  if (lig == (BWD ? GW - 1 : 0)) exc = aff_identity<V>();

  const V carry = row < g.E ? est.row_carry(row) : V(0);
  V A;
  if constexpr (NWR > 1) {
    Aff<V>* x = xw + rloc * NWR;
    if (lane == (BWD ? 0 : 31)) x[wr] = inc;
    __syncthreads();
    Aff<V> tw = lane < NWR ? x[lane] : aff_identity<V>();
#pragma unroll
    for (int off = 1; off < NWR; off <<= 1) {
      if (BWD) {
        Aff<V> o = shfl_down_aff(tw, off, 32);
        if (lane + off < NWR) tw = compose(tw, o);
      } else {
        Aff<V> o = shfl_up_aff(tw, off, 32);
        if (lane >= off) tw = compose(tw, o);
      }
    }
    const int src = BWD ? wr + 1 : wr - 1;
    Aff<V> ex = shfl_idx_aff(tw, src & 31, 32);
    if (BWD ? (wr == NWR - 1) : (wr == 0)) ex = aff_identity<V>();
    const V bval = ex.a + ex.b * carry;
    A = exc.a + exc.b * bval;
  } else {
    A = exc.a + exc.b * carry;
  }

  if (BWD) {
#pragma unroll
    for (int k = L - 1; k >= 0; --k) {
      V adj = A;
      A = c[k].a + c[k].b * A;
      est.emit(R, k, A, adj, c[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) {
      V adj = A;
      A = c[k].a + c[k].b * A;
      est.emit(R, k, A, adj, c[k]);
    }
  }
}

// ---------------------------------------------------------------------------
// fast env-major driver: the common case compiled without run-time
// generality.  Preconditions (checked by the planner): 16-byte aligned rows,
// T % LS == 0 and T <= TILE (one tile per row), one segment, one pass.
// A thread therefore holds either all LS steps or none, and a thread
// beyond its row's end contributes the identity map to the scan.
// ---------------------------------------------------------------------------
// Resident CTAs the fast env-major driver is compiled for.  One launch of a
// short-row workload (4096 x 128: 1024 CTAs of 128 threads) fills about half
// of the GPU's thread slots; consecutive launches overlap (the dependent
// grid launches as soon as this one has started, see pdl_trigger) only as
// far as the slots the running grid leaves free.  At 4 steps a thread the
// estimators fit 32 registers (at most a few bytes spilled), which makes
// every thread slot usable: 16 CTAs of 128 threads per SM.  Retrace (its
// action-axis staging), V-Trace with truncation and the 8-step variants
// spill tens to hundreds of bytes at 32 and keep the compiler's choice;
// V-Trace without truncation fits with 20 bytes spilled but measured slower
// capped in plain stream order (4096 x 256: 0.60 against 0.66 of the
// bandwidth) and is left uncapped unless RLCA_EM_CAP_VTRACE is set.
#ifndef RLCA_EM_CAP_VTRACE
#define RLCA_EM_CAP_VTRACE 0
#endif
// threads an SM the driver is compiled to keep resident at 4 steps a
// thread (0: the compiler's choice)
template <class Est>
struct EmRegCap {
  static constexpr int threads = 2048;
};
template <bool H, class ST>
struct EmRegCap<RetraceEst<H, ST>> {
  static constexpr int threads = 0;
};
template <class ST>
struct EmRegCap<VtraceEst<true, ST>> {
  static constexpr int threads = 0;
};
template <class ST>
struct EmRegCap<VtraceEst<false, ST>> {
  static constexpr int threads = RLCA_EM_CAP_VTRACE == 1 ? 2048 : (RLCA_EM_CAP_VTRACE == 2 ? 1536 : 0);
};
template <class Est, int BLOCK, int LS>
__host__ __device__ constexpr int em_fast_min_blocks() {
  return (EmRegCap<Est>::threads > 0 && LS == 4 && EmRegCap<Est>::threads >= BLOCK) ? EmRegCap<Est>::threads / BLOCK
                                                                                     : 1;
}

template <class Est, int TPR, int LS>
__global__ void __launch_bounds__(EmShape<TPR, LS>::BLOCK, (em_fast_min_blocks<Est, EmShape<TPR, LS>::BLOCK, LS>()))
    em_fast_kernel(Est est, Geom g) {
  using S = EmShape<TPR, LS>;
  using V = typename Est::V;
  constexpr int L = S::L, NWR = S::NWR;

  extern __shared__ __align__(16) unsigned char smem[];
  Aff<V>* xw = reinterpret_cast<Aff<V>*>(smem);  // [ROWS][NWR] warp totals (NWR > 1)
  unsigned char* est_smem = smem + (NWR > 1 ? 2 * S::ROWS * NWR * sizeof(Aff<V>) : 0);

  const int tid = threadIdx.x;
  const int j = tid % TPR;
  const int rloc = tid / TPR;
  const int64_t row0 = (int64_t)blockIdx.x * S::ROWS;
  const int64_t row = row0 + rloc;
  const int t0 = j * L;
  const bool active = row < g.E && t0 < g.T;
  const int n = active ? L : 0;
  const EnvMajor lay{g.E, g.T};
  const bool early = g.early != 0;
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (!early) pdl_wait();

  est.template stage<S::ROWS, S::BLOCK, S::TILE>(lay, g, row0, rloc, 0, g.T, est_smem);
  typename Est::template Regs<L> R;
  const GIO<EnvMajor, true, typename Est::Store> io{lay, row, t0, n, true};
  est.template load<L>(R, io, rloc, 0, S::TILE, S::ROWS, est_smem);

  em_fast_scan<Est, TPR, LS>(est, R, g, lay, row, t0, active, rloc, xw);
  if (early) pdl_wait();  // the previous kernel may still read or write what we overwrite
  if (active) est.template store<L>(R, io);
}

// ---------------------------------------------------------------------------
// time-major driver
// ---------------------------------------------------------------------------
template <class Est, int C>
__global__ void __launch_bounds__(TmShape<C>::BLOCK)
    tm_scan_kernel(Est est, Geom g) {
  using S = TmShape<C>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  constexpr int L = S::L;

  extern __shared__ __align__(16) unsigned char smem[];
  Aff<V>* xs = reinterpret_cast<Aff<V>*>(smem);  // [2][C][32] chunk maps
  unsigned char* est_smem = smem + 2 * C * 32 * sizeof(Aff<V>);

  const int lane = threadIdx.x & 31;
  const int cw = threadIdx.x >> 5;  // chunk index inside the tile
  const int seg = g.nseg == 1 ? 0 : (int)(blockIdx.x % (unsigned)g.nseg);
  const int64_t row0 = (int64_t)(g.nseg == 1 ? blockIdx.x : blockIdx.x / (unsigned)g.nseg) * S::EW;
  const int64_t row = row0 + lane;
  const bool row_ok = row < g.E;
  const int seg_lo = seg * g.seg_len;
  const int seg_hi = min(g.T, seg_lo + g.seg_len);
  const bool agg_mode = g.mode == kModeAggregate;
  const TimeMajor lay{g.E, g.T};
  const bool early = g.early != 0 && g.nseg == 1 && !agg_mode;
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (!early) pdl_wait();

  Aff<V> carry;
  if (agg_mode) {
    carry = aff_identity<V>();
  } else {
    V c0 = row_ok ? est.row_carry(row) : V(0);
    if (g.nseg > 1 && row_ok) c0 = segment_carry_in<V, BWD>(g, row, seg, c0);
    carry = {c0, V(0)};
  }

  const int ntiles = (seg_hi - seg_lo + S::TILE - 1) / S::TILE;
  for (int it = 0; it < ntiles; ++it) {
    const int tile = BWD ? ntiles - 1 - it : it;
    const int ts = seg_lo + tile * S::TILE;
    const int te = min(seg_hi, ts + S::TILE);
    const int t0 = ts + cw * L;
    const int n = row_ok ? max(0, min(L, te - t0)) : 0;

    est.template stage_tm<S::BLOCK>(lay, g, row0, ts, te, est_smem);
    typename Est::template Regs<L> R;
    const GIO<TimeMajor, false, typename Est::Store> io{lay, row, t0, n, false};
    est.template load<L>(R, io, lane, ts, S::TILE, 32, est_smem);
    if constexpr (Est::kNb > 0) {
      float got[Est::kNb > 0 ? Est::kNb : 1];
#pragma unroll
      for (int i = 0; i < Est::kNb; ++i) got[i] = 0.f;
      const int tn = BWD ? t0 + L : t0 - 1;
      if (n > 0 && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T)) est.nb_load(lay, row, tn, got);
      est.nb_take(R, got);
    }

    Aff<V> c[L];
#pragma unroll
    for (int k = 0; k < L; ++k) c[k] = (k < n) ? est.coef(R, k, t0 + k) : aff_identity<V>();
    Aff<V> agg = aff_identity<V>();
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) agg = compose(c[k], agg);
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) agg = compose(c[k], agg);
    }

    Aff<V>* x = xs + (it & 1) * C * 32;
    x[cw * 32 + lane] = agg;
    __syncthreads();
    Aff<V> cc = carry, boundary = carry;
    if (BWD) {
#pragma unroll 4
      for (int w = C - 1; w >= 0; --w) {
        if (w == cw) boundary = cc;
        cc = compose(x[w * 32 + lane], cc);
      }
    } else {
#pragma unroll 4
      for (int w = 0; w < C; ++w) {
        if (w == cw) boundary = cc;
        cc = compose(x[w * 32 + lane], cc);
      }
    }

    if (!agg_mode) {
      V A = boundary.a;
      if (BWD) {
#pragma unroll
        for (int k = L - 1; k >= 0; --k) {
          V adj = A;
          A = c[k].a + c[k].b * A;
          est.emit(R, k, A, adj, c[k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < L; ++k) {
          V adj = A;
          A = c[k].a + c[k].b * A;
          est.emit(R, k, A, adj, c[k]);
        }
      }
      if (early && it == 0) pdl_wait();
      est.template store<L>(R, io);
    }
    carry = cc;
  }
  if (agg_mode && row_ok && cw == 0 && in_range(row * g.nseg + seg, g.E * (int64_t)g.nseg))
    reinterpret_cast<Aff<V>*>(g.ws)[row * g.nseg + seg] = carry;
}

// ---------------------------------------------------------------------------
// fast time-major driver.  Preconditions (checked by the planner): T % L == 0,
// E * T < 2^32; few environments with long rows run it as the two-pass
// segmented split (segment maps, then the segments from their entering
// values), like the general drivers.  Each tile of CT * L steps: every
// thread composes its chunk's L maps from coalesced step rows (EW
// consecutive environments per load), the CT chunk maps of an environment are
// scanned by CT adjacent lanes with shuffles (log2 CT rounds instead of a
// serial walk), and the chunk boundary values come back through shared
// memory.  The scan lanes of an environment keep its carry across tiles.
// ---------------------------------------------------------------------------
// the 64-register cap of the fast time-major drivers pays where a kernel
// needs only a few more; the staged V-Trace needs ~80 and runs faster
// uncapped than spilling (its direct sibling is faster capped)
template <class Est>
struct TfRegCap {
  static constexpr bool value = true;
};
template <bool H, class ST>
struct TfRegCap<VtraceEst<H, ST>> {
  static constexpr bool value = false;
};
template <class Est, int BLOCK>
__host__ __device__ constexpr int tf_blocks_for() {
  return TfRegCap<Est>::value ? tf_min_blocks(BLOCK) : 1;
}

template <class Est, int EW, int CT>
__global__ void __launch_bounds__(TfShape<EW, CT>::BLOCK, tf_min_blocks(TfShape<EW, CT>::BLOCK))
    tm_fast_kernel(Est est, Geom g) {
  using S = TfShape<EW, CT>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  constexpr int L = S::L, PAD = S::PAD;

  extern __shared__ __align__(16) unsigned char smem[];
  Aff<V>* xs = reinterpret_cast<Aff<V>*>(smem);  // [CT][PAD] chunk maps
  V* ys = reinterpret_cast<V*>(xs + CT * PAD);    // [CT][PAD] values entering each chunk

  const int tid = threadIdx.x;
  const int j = tid % EW, c = tid / EW;    // load / emit role
  const int js = tid / CT, cs = tid % CT;  // scan role
  const int seg = g.nseg == 1 ? 0 : (int)(blockIdx.x % (unsigned)g.nseg);
  const int64_t row0 = (int64_t)(g.nseg == 1 ? blockIdx.x : blockIdx.x / (unsigned)g.nseg) * EW;
  const int64_t row = row0 + j;
  const bool row_ok = row < g.E;
  const int seg_lo = seg * g.seg_len;
  const int seg_hi = min(g.T, seg_lo + g.seg_len);
  const bool agg_mode = g.mode == kModeAggregate;
  const uint32_t E32 = (uint32_t)g.E;
  const TimeMajor lay{g.E, g.T};
  const bool early = g.early != 0 && g.nseg == 1;
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (!early) pdl_wait();

  // scan role: the value entering this segment (full pass) or the map of
  // the whole segment (first pass of the two-pass path)
  V carry = V(0);
  Aff<V> seg_map = aff_identity<V>();
  if (!agg_mode && row0 + js < g.E) {
    carry = est.row_carry(row0 + js);
    if (g.nseg > 1) carry = segment_carry_in<V, BWD>(g, row0 + js, seg, carry);
  }
  const int ntiles = (seg_hi - seg_lo + S::TILE - 1) / S::TILE;
  for (int it = 0; it < ntiles; ++it) {
    const int tile = BWD ? ntiles - 1 - it : it;
    const int ts = seg_lo + tile * S::TILE;
    const int t0 = ts + c * L;
    const int n = (row_ok && t0 < seg_hi) ? L : 0;
    const TmIO32<typename Est::Store> io{row, t0, n, (uint32_t)t0 * E32 + (uint32_t)row, E32,
                                               E32 * (uint32_t)g.T};

    typename Est::template Regs<L> R;
    est.template load<L>(R, io, 0, ts, S::TILE, EW, nullptr);
    if constexpr (Est::kNb > 0) {
      float got[Est::kNb > 0 ? Est::kNb : 1];
#pragma unroll
      for (int i = 0; i < Est::kNb; ++i) got[i] = 0.f;
      const int tn = BWD ? t0 + L : t0 - 1;
      if (n > 0 && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T)) est.nb_load(lay, row, tn, got);
      est.nb_take(R, got);
    }

    Aff<V> cf[L];
#pragma unroll
    for (int k = 0; k < L; ++k) cf[k] = n != 0 ? est.coef(R, k, t0 + k) : aff_identity<V>();
    Aff<V> agg = aff_identity<V>();
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) agg = compose(cf[k], agg);
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) agg = compose(cf[k], agg);
    }
    xs[c * PAD + j] = agg;
    __syncthreads();

    // scan role: inclusive scan of environment js's chunk maps in time order
    // of application (suffix for a backward scan, prefix for a forward one)
    Aff<V> m = xs[cs * PAD + js];
#pragma unroll
    for (int d = 1; d < CT; d <<= 1) {
      if (BWD) {
        const Aff<V> o = shfl_down_aff(m, d, CT);
        if (cs + d < CT) m = compose(m, o);
      } else {
        const Aff<V> o = shfl_up_aff(m, d, CT);
        if (cs >= d) m = compose(m, o);
      }
    }
    Aff<V> ex = BWD ? shfl_down_aff(m, 1, CT) : shfl_up_aff(m, 1, CT);
    if (cs == (BWD ? CT - 1 : 0)) ex = aff_identity<V>();
    const Aff<V> tot = shfl_idx_aff(m, BWD ? 0 : CT - 1, CT);
    if (agg_mode) {
      seg_map = compose(tot, seg_map);  // tiles arrive in the order the recurrence applies them
    } else {
      ys[cs * PAD + js] = ex.a + ex.b * carry;
      carry = tot.a + tot.b * carry;
    }
    __syncthreads();
    if (agg_mode) continue;

    V A = ys[c * PAD + j];
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    }
    if (early && it == 0) pdl_wait();  // the previous kernel may still read or write what we overwrite
    est.template store<L>(R, io);
  }
  if (agg_mode && cs == 0 && row0 + js < g.E && in_range((row0 + js) * g.nseg + seg, g.E * (int64_t)g.nseg))
    reinterpret_cast<Aff<V>*>(g.ws)[(row0 + js) * g.nseg + seg] = seg_map;
}

// ---------------------------------------------------------------------------
// staged time-major driver.  Preconditions: those of the fast time-major
// driver (the two-pass split included), E a multiple of the environments of
// a 16-byte piece, 16-byte aligned float inputs and 4-byte aligned flag
// inputs.  The inputs of the tiles stream into a ring of NS shared-memory
// stages with cp.async (16-byte pieces of a step row for floats, 4-byte
// pieces for flags), NS - 1 tiles ahead of the tile being scanned, so the
// bytes in flight depend on neither registers nor occupancy.  The scan is
// the fast time-major one; outputs go straight to global memory.
// ---------------------------------------------------------------------------
template <class Est, int EW, int CT>
__global__ void __launch_bounds__(TsShape<EW, CT>::BLOCK, (tf_blocks_for<Est, TsShape<EW, CT>::BLOCK>()))
    tm_staged_kernel(Est est, Geom g) {
  using S = TsShape<EW, CT>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  using ST = typename Est::Store;
  constexpr int L = S::L, PAD = S::PAD, NS = S::NS, CS = S::CS, FB = S::FB;
  constexpr int ES = (int)sizeof(ST);
  constexpr int FPE = 16 / ES;              // environments per 16-byte piece of a float row
  constexpr int QF = EW / FPE;              // float pieces per step row
  constexpr int QB = EW / 4;                // 4-byte flag pieces per step row
  constexpr int PF = S::TILE * QF;          // float pieces per staged input and tile
  constexpr int PB = S::TILE * QB;          // flag pieces per staged input and tile
  constexpr size_t STAGE = ts_stage_bytes<Est, EW, CT>();
  constexpr size_t FLAGS_AT = (size_t)ES * Est::kSF * FB;  // flag buffers' offset in a stage
  static_assert(PF % S::BLOCK == 0 && PB % S::BLOCK == 0, "whole copy rounds");

  extern __shared__ __align__(16) unsigned char smem[];
  Aff<V>* xs = reinterpret_cast<Aff<V>*>(smem);  // [CT][PAD] chunk maps
  V* ys = reinterpret_cast<V*>(xs + CT * PAD);    // [CT][PAD] values entering each chunk
  unsigned char* ring = smem + align16(tf_smem_bytes<V, EW, CT>());

  const int tid = threadIdx.x;
  const int j = tid % EW, c = tid / EW;    // load / emit role
  const int js = tid / CT, cs = tid % CT;  // scan role
  const int seg = g.nseg == 1 ? 0 : (int)(blockIdx.x % (unsigned)g.nseg);
  const int64_t row0 = (int64_t)(g.nseg == 1 ? blockIdx.x : blockIdx.x / (unsigned)g.nseg) * EW;
  const int64_t row = row0 + j;
  const bool row_ok = row < g.E;
  const int seg_lo = seg * g.seg_len;
  const int seg_hi = min(g.T, seg_lo + g.seg_len);
  const bool agg_mode = g.mode == kModeAggregate;
  const uint32_t E32 = (uint32_t)g.E;
  const uint32_t e0 = (uint32_t)row0;
  const TimeMajor lay{g.E, g.T};
  const bool early = g.early != 0 && g.nseg == 1;
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (!early) pdl_wait();

  StagedList in;
  est.staged_io(in);
  const int ntiles = (seg_hi - seg_lo + S::TILE - 1) / S::TILE;

  // issue the copies of the it-th tile in processing order into stage it % NS
  // (one commit group per call, empty past the last tile)
  auto stage_tile = [&](int it) {
    if (it < ntiles) {
      const int ts = seg_lo + (BWD ? ntiles - 1 - it : it) * S::TILE;
      unsigned char* st = ring + (size_t)(it % NS) * STAGE;
      // float inputs: 16-byte pieces of FPE environments (E % FPE == 0: a
      // piece is wholly inside or outside the rows)
#pragma unroll
      for (int i = 0; i < PF / S::BLOCK; ++i) {
        const int p = tid + i * S::BLOCK;
        const int r = p / QF, q = p % QF;
        const int t = ts + r;
        const uint32_t e = e0 + (uint32_t)(FPE * q);
        if (t < g.T && e < E32) {
          const uint32_t go = (uint32_t)t * E32 + e;
          const int so = (r / L) * CS + (r % L) * EW + FPE * q;
          if (span_in_range(go, FPE, (int64_t)E32 * g.T) && span_in_range(so, FPE, FB)) {
#pragma unroll
            for (int b = 0; b < Est::kSF; ++b)
              cp_async16(reinterpret_cast<ST*>(st) + b * FB + so, static_cast<const ST*>(in.fin[b]) + go);
          }
        }
      }
      // flag inputs: 4-byte pieces of 4 environments
#pragma unroll
      for (int i = 0; i < PB / S::BLOCK; ++i) {
        const int p = tid + i * S::BLOCK;
        const int r = p / QB, q = p % QB;
        const int t = ts + r;
        const uint32_t e = e0 + 4u * (uint32_t)q;
        if (t < g.T && e < E32) {
          const uint32_t go = (uint32_t)t * E32 + e;
          const int so = (r / L) * CS + (r % L) * EW + 4 * q;
          if (span_in_range(go, 4, (int64_t)E32 * g.T) && span_in_range(so, 4, FB)) {
#pragma unroll
            for (int b = 0; b < Est::kSB; ++b)
              if (in.bin[b] != nullptr) cp_async4(st + FLAGS_AT + b * FB + so, in.bin[b] + go);
          }
        }
      }
    }
    cp_async_commit();
  };

  // the neighbour step's inputs of the it-th tile, loaded one tile ahead
  constexpr int NB = Est::kNb > 0 ? Est::kNb : 1;
  auto nb_fetch = [&](int it, float (&got)[NB]) {
#pragma unroll
    for (int i = 0; i < NB; ++i) got[i] = 0.f;
    if (Est::kNb > 0 && it < ntiles) {
      const int t0 = seg_lo + (BWD ? ntiles - 1 - it : it) * S::TILE + c * L;
      const int tn = BWD ? t0 + L : t0 - 1;
      if (row_ok && t0 < seg_hi && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T))
        est.nb_load(lay, row, tn, got);
    }
  };

#pragma unroll
  for (int s = 0; s < NS - 1; ++s) stage_tile(s);
  float nb_cur[NB];
  nb_fetch(0, nb_cur);
  cp_async_wait<NS - 2>();
  __syncthreads();

  // scan role: the value entering this segment (full pass) or the map of
  // the whole segment (first pass of the two-pass path)
  V carry = V(0);
  Aff<V> seg_map = aff_identity<V>();
  if (!agg_mode && row0 + js < g.E) {
    carry = est.row_carry(row0 + js);
    if (g.nseg > 1) carry = segment_carry_in<V, BWD>(g, row0 + js, seg, carry);
  }
  for (int it = 0; it < ntiles; ++it) {
    stage_tile(it + NS - 1);  // into the stage every thread finished reading in iteration it - 1
    float nb_nxt[NB];
    nb_fetch(it + 1, nb_nxt);
    const int tile = BWD ? ntiles - 1 - it : it;
    const int ts = seg_lo + tile * S::TILE;
    const int t0 = ts + c * L;
    const int n = (row_ok && t0 < seg_hi) ? L : 0;
    const unsigned char* st = ring + (size_t)(it % NS) * STAGE;
    const TmSIO<EW, FB, ST> io{reinterpret_cast<const ST*>(st), st + FLAGS_AT, c * CS + j, c * CS + j, row, t0, n,
                               (uint32_t)t0 * E32 + (uint32_t)row, E32, E32 * (uint32_t)g.T};

    typename Est::template Regs<L> R;
    est.template load<L>(R, io, 0, ts, S::TILE, EW, nullptr);
    if constexpr (Est::kNb > 0) est.nb_take(R, nb_cur);
#pragma unroll
    for (int i = 0; i < NB; ++i) nb_cur[i] = nb_nxt[i];

    Aff<V> cf[L];
#pragma unroll
    for (int k = 0; k < L; ++k) cf[k] = n != 0 ? est.coef(R, k, t0 + k) : aff_identity<V>();
    Aff<V> agg = aff_identity<V>();
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) agg = compose(cf[k], agg);
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) agg = compose(cf[k], agg);
    }
    xs[c * PAD + j] = agg;
    __syncthreads();

    Aff<V> m = xs[cs * PAD + js];
#pragma unroll
    for (int d = 1; d < CT; d <<= 1) {
      if (BWD) {
        const Aff<V> o = shfl_down_aff(m, d, CT);
        if (cs + d < CT) m = compose(m, o);
      } else {
        const Aff<V> o = shfl_up_aff(m, d, CT);
        if (cs >= d) m = compose(m, o);
      }
    }
    Aff<V> ex = BWD ? shfl_down_aff(m, 1, CT) : shfl_up_aff(m, 1, CT);
    if (cs == (BWD ? CT - 1 : 0)) ex = aff_identity<V>();
    const Aff<V> tot = shfl_idx_aff(m, BWD ? 0 : CT - 1, CT);
    if (agg_mode) {
      seg_map = compose(tot, seg_map);  // tiles arrive in the order the recurrence applies them
    } else {
      ys[cs * PAD + js] = ex.a + ex.b * carry;
      carry = tot.a + tot.b * carry;
    }
    cp_async_wait<NS - 2>();  // this thread's copies of tile it + 1 have landed
    __syncthreads();          // ... everyone's, and the chunk entry values are visible
    if (agg_mode) continue;

    V A = ys[c * PAD + j];
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    }
    if (early && it == 0) pdl_wait();  // the previous kernel may still read or write what we overwrite
    est.template store<L>(R, io);
  }
  if (agg_mode && cs == 0 && row0 + js < g.E && in_range((row0 + js) * g.nseg + seg, g.E * (int64_t)g.nseg))
    reinterpret_cast<Aff<V>*>(g.ws)[(row0 + js) * g.nseg + seg] = seg_map;
}

// ---------------------------------------------------------------------------
// bulk time-major driver: the staged driver's tile loop with each tile's
// inputs moved by the tensor memory accelerator.  Preconditions (checked by
// the planner): T % 8 == 0, E * T < 2^32, E % 16 == 0, 16-byte aligned
// inputs, one 2-D tensor map per staged input (TmaSet, encoded on the host).
// Per tile and input, thread 0 issues one cp.async.bulk.tensor copy of the
// [TILE, EW] block into a ring of NS stages, NS - 1 tiles ahead of the scan;
// completion is counted in bytes on the stage's mbarrier.  A copy's rows
// are at least 16 bytes wide: CTAs of 8 environments copy the flag rows of
// the aligned 16 environments that hold theirs and read their half.  No
// thread issues
// per-element copies, so the bytes in flight are set by the ring, not by
// registers or occupancy.  Every wait is bounded (mbar_wait_bounded): a
// copy that never lands sets the status word and the CTA returns.
// ---------------------------------------------------------------------------
#ifndef RLCA_TB_STAGES
#define RLCA_TB_STAGES 2
#endif
template <int EW, int CT>
struct TbShape : TfShape<EW, CT> {
  static constexpr int NS = RLCA_TB_STAGES;
  static constexpr int CS = TfShape<EW, CT>::L * EW;  // chunk stride in a stage buffer: [TILE][EW], dense
  static constexpr int FB = CT * CS;                  // elements per staged buffer (= TILE * EW)
  static constexpr int FW = EW < 16 ? 16 : EW;        // bytes per staged flag row (16 at least)
  static constexpr int FBB = TfShape<EW, CT>::TILE * FW;  // bytes per staged flag buffer
  static_assert(EW == 8 || EW == 16 || EW == 32, "float rows of 32 bytes or more");
};
template <class Est, int EW, int CT>
__host__ __device__ constexpr size_t tb_stage_bytes() {
  // FB * element size and FBB are multiples of 128 (TILE % 8 == 0, rows of
  // >= 16 bytes), so every buffer starts on a 128-byte boundary
  return (size_t)TbShape<EW, CT>::FB * sizeof(typename Est::Store) * Est::kSF +
         (size_t)TbShape<EW, CT>::FBB * Est::kSB;
}
template <class Est, int EW, int CT>
__host__ __device__ constexpr size_t tb_smem_bytes() {
  // barriers (128 B), exchange arrays, up to 128 B of alignment slack, ring
  return 128 + align16(tf_smem_bytes<typename Est::V, EW, CT>()) + 128 +
         TbShape<EW, CT>::NS * tb_stage_bytes<Est, EW, CT>();
}

template <class Est, int EW, int CT>
__global__ void __launch_bounds__(TbShape<EW, CT>::BLOCK, (tf_blocks_for<Est, TbShape<EW, CT>::BLOCK>()))
    tm_bulk_kernel(Est est, Geom g, const __grid_constant__ TmaSet maps) {
  using S = TbShape<EW, CT>;
  using V = typename Est::V;
  constexpr bool BWD = Est::kBackward;
  using ST = typename Est::Store;
  constexpr int L = S::L, PAD = S::PAD, NS = S::NS, CS = S::CS, FB = S::FB, FW = S::FW, FBB = S::FBB;
  constexpr int ES = (int)sizeof(ST);
  constexpr size_t STAGE = tb_stage_bytes<Est, EW, CT>();
  constexpr size_t FLAGS_AT = (size_t)ES * Est::kSF * FB;  // flag buffers' offset in a stage

  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);         // [NS] stage barriers
  int* abort_flag = reinterpret_cast<int*>(smem + 8 * NS);    // set by a wait that gave up
  Aff<V>* xs = reinterpret_cast<Aff<V>*>(smem + 128);        // [CT][PAD] chunk maps
  V* ys = reinterpret_cast<V*>(xs + CT * PAD);                // [CT][PAD] values entering each chunk
  const uintptr_t rb = reinterpret_cast<uintptr_t>(smem + 128 + align16(tf_smem_bytes<V, EW, CT>()));
  unsigned char* ring = reinterpret_cast<unsigned char*>((rb + 127) & ~uintptr_t(127));

  const int tid = threadIdx.x;
  const int j = tid % EW, c = tid / EW;    // load / emit role
  const int js = tid / CT, cs = tid % CT;  // scan role
  const int seg = g.nseg == 1 ? 0 : (int)(blockIdx.x % (unsigned)g.nseg);
  const int64_t row0 = (int64_t)(g.nseg == 1 ? blockIdx.x : blockIdx.x / (unsigned)g.nseg) * EW;
  const int64_t row = row0 + j;
  const bool row_ok = row < g.E;
  const int seg_lo = seg * g.seg_len;
  const int seg_hi = min(g.T, seg_lo + g.seg_len);
  const bool agg_mode = g.mode == kModeAggregate;
  const uint32_t E32 = (uint32_t)g.E;
  const TimeMajor lay{g.E, g.T};
  const bool early = g.early != 0 && g.nseg == 1;
  // flag rows: copied from environment fx (16-byte aligned), ours at foff
  const int fx = EW < 16 ? (int)(row0 & ~int64_t(15)) : (int)row0;
  const int foff = (int)(row0 - fx);
  pdl_trigger();  // the dependent grid may launch now: it waits for this one before touching our outputs
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bars[s], 1);
    *abort_flag = 0;
    mbar_fence_init();
#pragma unroll
    for (int b = 0; b < Est::kSF; ++b) tma_prefetch_map(&maps.f[b]);
  }
  if (!early) pdl_wait();
  __syncthreads();

  StagedList in;
  est.staged_io(in);
  const int ntiles = (seg_hi - seg_lo + S::TILE - 1) / S::TILE;
  int nflags = 0;
#pragma unroll
  for (int b = 0; b < Est::kSB; ++b) nflags += in.bin[b] != nullptr ? 1 : 0;
  const uint32_t tx_bytes = (uint32_t)(S::TILE * EW * ES * Est::kSF) + (uint32_t)(FBB * nflags);

  // thread 0: the copies of the it-th tile in processing order into stage it % NS
  auto issue = [&](int it) {
    if (it >= ntiles) return;
    const int ts = seg_lo + (BWD ? ntiles - 1 - it : it) * S::TILE;
    unsigned char* st = ring + (size_t)(it % NS) * STAGE;
    uint64_t* bar = &bars[it % NS];
    mbar_arrive_expect_tx(bar, tx_bytes);
#pragma unroll
    for (int b = 0; b < Est::kSF; ++b) tma_load_2d(st + (size_t)b * FB * ES, &maps.f[b], (int)row0, ts, bar);
#pragma unroll
    for (int b = 0; b < Est::kSB; ++b)
      if (in.bin[b] != nullptr) tma_load_2d(st + FLAGS_AT + (size_t)b * FBB, &maps.b[b], fx, ts, bar);
  };
  // thread 0, after a wait gave up: let the copies already issued land (each
  // wait bounded again) before the CTA exits
  auto drain = [&](int from) {
    for (int k = from; k < ntiles && k < from + NS; ++k) mbar_wait_bounded(&bars[k % NS], (uint32_t)(k / NS) & 1u);
  };

  // the neighbour step's inputs of the it-th tile, loaded one tile ahead
  constexpr int NB = Est::kNb > 0 ? Est::kNb : 1;
  auto nb_fetch = [&](int it, float (&got)[NB]) {
#pragma unroll
    for (int i = 0; i < NB; ++i) got[i] = 0.f;
    if (Est::kNb > 0 && it < ntiles) {
      const int t0 = seg_lo + (BWD ? ntiles - 1 - it : it) * S::TILE + c * L;
      const int tn = BWD ? t0 + L : t0 - 1;
      if (row_ok && t0 < seg_hi && tn >= 0 && tn < g.T && in_range(lay.at(row, tn), g.E * (int64_t)g.T))
        est.nb_load(lay, row, tn, got);
    }
  };

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) issue(s);
  }
  float nb_cur[NB];
  nb_fetch(0, nb_cur);

  // scan role: the value entering this segment (full pass) or the map of
  // the whole segment (first pass of the two-pass path)
  V carry = V(0);
  Aff<V> seg_map = aff_identity<V>();
  if (!agg_mode && row0 + js < g.E) {
    carry = est.row_carry(row0 + js);
    if (g.nseg > 1) carry = segment_carry_in<V, BWD>(g, row0 + js, seg, carry);
  }
  for (int it = 0; it < ntiles; ++it) {
    // stage (it - 1) % NS was last read before the first barrier of iteration it - 1
    if (tid == 0) issue(it + NS - 1);
    float nb_nxt[NB];
    nb_fetch(it + 1, nb_nxt);
    const int tile = BWD ? ntiles - 1 - it : it;
    const int ts = seg_lo + tile * S::TILE;
    const int t0 = ts + c * L;
    const int n = (row_ok && t0 < seg_hi) ? L : 0;
    const unsigned char* st = ring + (size_t)(it % NS) * STAGE;
    if (!mbar_wait_bounded(&bars[it % NS], (uint32_t)(it / NS) & 1u)) *abort_flag = 1;
    const TmSIO<EW, FB, ST, FW, FBB> io{reinterpret_cast<const ST*>(st), st + FLAGS_AT, c * CS + j,
                                        c * L * FW + foff + j, row, t0, n, (uint32_t)t0 * E32 + (uint32_t)row,
                                        E32, E32 * (uint32_t)g.T};

    typename Est::template Regs<L> R;
    est.template load<L>(R, io, 0, ts, S::TILE, EW, nullptr);
    if constexpr (Est::kNb > 0) est.nb_take(R, nb_cur);
#pragma unroll
    for (int i = 0; i < NB; ++i) nb_cur[i] = nb_nxt[i];

    Aff<V> cf[L];
#pragma unroll
    for (int k = 0; k < L; ++k) cf[k] = n != 0 ? est.coef(R, k, t0 + k) : aff_identity<V>();
    Aff<V> agg = aff_identity<V>();
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) agg = compose(cf[k], agg);
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) agg = compose(cf[k], agg);
    }
    xs[c * PAD + j] = agg;
    __syncthreads();
    if (*abort_flag != 0) {  // uniform: read after the barrier by every thread
      if (tid == 0) drain(it);
      return;
    }

    Aff<V> m = xs[cs * PAD + js];
#pragma unroll
    for (int d = 1; d < CT; d <<= 1) {
      if (BWD) {
        const Aff<V> o = shfl_down_aff(m, d, CT);
        if (cs + d < CT) m = compose(m, o);
      } else {
        const Aff<V> o = shfl_up_aff(m, d, CT);
        if (cs >= d) m = compose(m, o);
      }
    }
    Aff<V> ex = BWD ? shfl_down_aff(m, 1, CT) : shfl_up_aff(m, 1, CT);
    if (cs == (BWD ? CT - 1 : 0)) ex = aff_identity<V>();
    const Aff<V> tot = shfl_idx_aff(m, BWD ? 0 : CT - 1, CT);
    if (agg_mode) {
      seg_map = compose(tot, seg_map);  // tiles arrive in the order the recurrence applies them
    } else {
      ys[cs * PAD + js] = ex.a + ex.b * carry;
      carry = tot.a + tot.b * carry;
    }
    __syncthreads();
    if (agg_mode) continue;

    V A = ys[c * PAD + j];
    if (BWD) {
#pragma unroll
      for (int k = L - 1; k >= 0; --k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < L; ++k) {
        V adj = A;
        A = cf[k].a + cf[k].b * A;
        est.emit(R, k, A, adj, cf[k]);
      }
    }
    if (early && it == 0) pdl_wait();  // the previous kernel may still read or write what we overwrite
    est.template store<L>(R, io);
  }
  if (agg_mode && cs == 0 && row0 + js < g.E && in_range((row0 + js) * g.nseg + seg, g.E * (int64_t)g.nseg))
    reinterpret_cast<Aff<V>*>(g.ws)[(row0 + js) * g.nseg + seg] = seg_map;
}



}  // namespace rlca
