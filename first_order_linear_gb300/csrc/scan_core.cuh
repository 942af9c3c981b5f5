// scan_core.cuh -- device building blocks of the credit-assignment scans.
//
// The recurrence of rl-triton (arXiv:2608.17641) §1 Introduction,
//   backward  A_t = alpha_t + beta_t * A_{t+1},   forward  A_t = alpha_t + beta_t * A_{t-1},
// is evaluated with the paper's combine (§2.2 Associative Scan; the
// technical summary's (alpha_B, beta_B) (+) (alpha_A, beta_A) =
// (alpha_B + beta_B alpha_A, beta_A beta_B)): composing the affine maps
// x -> alpha + beta x.  Associativity (§5 Correctness Analysis) lets each
// level below regroup the same sequential product:
//
//   1. a thread composes its L consecutive steps serially in registers,
//   2. a warp scans the per-thread maps with log2(lanes) shuffle rounds
//      (the stride-1, stride-2, ... passes of Appendix A),
//   3. warps of one row exchange their totals through shared memory,
//   4. a row longer than one tile is walked tile by tile, the value at the
//      tile edge carried in a register,
//   5. rows split into segments across CTAs (two-pass path) get the value at
//      their segment edge from the per-segment maps of the first pass,
// and finally each thread re-expands its L steps from its incoming value.
//
// The same drivers serve every estimator: an estimator functor (see
// estimators.cuh) loads its raw inputs, builds (alpha_t, beta_t) in
// registers and writes its outputs.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rlca {

constexpr unsigned kFullMask = 0xffffffffu;

// x -> a + b * x
template <class V>
struct Aff {
  V a, b;
};

template <class V>
__device__ __forceinline__ Aff<V> aff_identity() {
  return {V(0), V(1)};
}

// outer o inner : x -> outer.a + outer.b * (inner.a + inner.b * x)
template <class V>
__device__ __forceinline__ Aff<V> compose(const Aff<V>& outer, const Aff<V>& inner) {
  return {outer.a + outer.b * inner.a, outer.b * inner.b};
}

// Three independent recurrences scanned side by side (the fused value-target
// scan: GAE, discounted return and TD(lambda) of one row).  Arithmetic is
// element-wise, so compose() on Aff<F3> composes the three maps at once.
struct F3 {
  float x, y, z;
  __host__ __device__ F3() = default;
  __host__ __device__ constexpr F3(float s) : x(s), y(s), z(s) {}
  __host__ __device__ constexpr F3(float a, float b, float c) : x(a), y(b), z(c) {}
};
__device__ __forceinline__ F3 operator+(const F3& a, const F3& b) { return {a.x + b.x, a.y + b.y, a.z + b.z}; }
__device__ __forceinline__ F3 operator*(const F3& a, const F3& b) { return {a.x * b.x, a.y * b.y, a.z * b.z}; }

__device__ __forceinline__ float shfl_down_v(float v, int d, int w) { return __shfl_down_sync(kFullMask, v, d, w); }
__device__ __forceinline__ uint32_t shfl_down_v(uint32_t v, int d, int w) {
  return __shfl_down_sync(kFullMask, v, d, w);
}
__device__ __forceinline__ F3 shfl_down_v(const F3& v, int d, int w) {
  return {shfl_down_v(v.x, d, w), shfl_down_v(v.y, d, w), shfl_down_v(v.z, d, w)};
}
__device__ __forceinline__ float shfl_up_v(float v, int d, int w) { return __shfl_up_sync(kFullMask, v, d, w); }
__device__ __forceinline__ uint32_t shfl_up_v(uint32_t v, int d, int w) { return __shfl_up_sync(kFullMask, v, d, w); }
__device__ __forceinline__ F3 shfl_up_v(const F3& v, int d, int w) {
  return {shfl_up_v(v.x, d, w), shfl_up_v(v.y, d, w), shfl_up_v(v.z, d, w)};
}
__device__ __forceinline__ float shfl_idx_v(float v, int s, int w) { return __shfl_sync(kFullMask, v, s, w); }
__device__ __forceinline__ uint32_t shfl_idx_v(uint32_t v, int s, int w) { return __shfl_sync(kFullMask, v, s, w); }
__device__ __forceinline__ F3 shfl_idx_v(const F3& v, int s, int w) {
  return {shfl_idx_v(v.x, s, w), shfl_idx_v(v.y, s, w), shfl_idx_v(v.z, s, w)};
}

template <class V>
__device__ __forceinline__ Aff<V> shfl_down_aff(const Aff<V>& x, int d, int w) {
  return {shfl_down_v(x.a, d, w), shfl_down_v(x.b, d, w)};
}
template <class V>
__device__ __forceinline__ Aff<V> shfl_up_aff(const Aff<V>& x, int d, int w) {
  return {shfl_up_v(x.a, d, w), shfl_up_v(x.b, d, w)};
}
template <class V>
__device__ __forceinline__ Aff<V> shfl_idx_aff(const Aff<V>& x, int src, int w) {
  return {shfl_idx_v(x.a, src, w), shfl_idx_v(x.b, src, w)};
}

// ---------------------------------------------------------------------------
// layouts: element index of (row e, step t)
// ---------------------------------------------------------------------------
struct EnvMajor {  // [E, T], t fastest
  static constexpr bool kTimeMajor = false;
  int64_t E;
  int T;
  __device__ __forceinline__ int64_t at(int64_t row, int t) const { return row * (int64_t)T + t; }
};
struct TimeMajor {  // [T, E], e fastest
  static constexpr bool kTimeMajor = true;
  int64_t E;
  int T;
  __device__ __forceinline__ int64_t at(int64_t row, int t) const { return (int64_t)t * E + row; }
};

// ---------------------------------------------------------------------------
// loads and stores of a thread's L consecutive steps
// ---------------------------------------------------------------------------
// vec: env-major rows are 16-byte aligned and T % 4 == 0, so a chunk of 4
// steps is one float4 (one u32 of flags) and is either fully in range or not.
template <int L, class Lay>
__device__ __forceinline__ void load_vals(const float* __restrict__ p, const Lay& lay, int64_t row,
                                          int t0, int n, bool vec, float (&out)[L]) {
  if (vec) {
    const float4* q = reinterpret_cast<const float4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i) {
      float4 v = (4 * i < n) ? __ldg(q + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      out[4 * i + 0] = v.x;
      out[4 * i + 1] = v.y;
      out[4 * i + 2] = v.z;
      out[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) out[k] = (k < n) ? __ldg(p + lay.at(row, t0 + k)) : 0.f;
  }
}

template <int L, class Lay>
__device__ __forceinline__ void load_ints(const int32_t* __restrict__ p, const Lay& lay, int64_t row,
                                          int t0, int n, bool vec, uint32_t (&out)[L]) {
  if (vec) {
    const int4* q = reinterpret_cast<const int4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i) {
      int4 v = (4 * i < n) ? __ldg(q + i) : make_int4(0, 0, 0, 0);
      out[4 * i + 0] = (uint32_t)v.x;
      out[4 * i + 1] = (uint32_t)v.y;
      out[4 * i + 2] = (uint32_t)v.z;
      out[4 * i + 3] = (uint32_t)v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) out[k] = (k < n) ? (uint32_t)__ldg(p + lay.at(row, t0 + k)) : 0u;
  }
}

// bit k of the result = (flag at step t0+k != 0); 0 for a NULL array
template <int L, class Lay>
__device__ __forceinline__ uint32_t load_flags(const uint8_t* __restrict__ p, const Lay& lay, int64_t row,
                                               int t0, int n, bool vec) {
  if (p == nullptr) return 0u;
  uint32_t bits = 0u;
  if (vec) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i) {
      const uint32_t w = (4 * i < n) ? __ldg(q + i) : 0u;
      // one bit per nonzero byte: bytes -> 0/1, then the multiply gathers
      // byte k's bit into bit 24 + k (the partial products never overlap)
      const uint32_t m = __vcmpne4(w, 0u) & 0x01010101u;
      bits |= ((m * 0x01020408u) >> 24) << (4 * i);
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) {
      if (k < n && __ldg(p + lay.at(row, t0 + k)) != 0) bits |= 1u << k;
    }
  }
  return bits;
}

template <class Lay>
__device__ __forceinline__ bool load_flag1(const uint8_t* __restrict__ p, const Lay& lay, int64_t row, int t) {
  return p != nullptr && __ldg(p + lay.at(row, t)) != 0;
}

template <int L, class Lay>
__device__ __forceinline__ void store_vals(float* __restrict__ p, const Lay& lay, int64_t row, int t0,
                                           int n, bool vec, const float (&v)[L]) {
  if (vec) {
    float4* q = reinterpret_cast<float4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i)
      if (4 * i < n) q[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (k < n) p[lay.at(row, t0 + k)] = v[k];
  }
}

template <int L, class Lay>
__device__ __forceinline__ void store_ints(int32_t* __restrict__ p, const Lay& lay, int64_t row, int t0,
                                           int n, bool vec, const uint32_t (&v)[L]) {
  if (vec) {
    int4* q = reinterpret_cast<int4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i)
      if (4 * i < n)
        q[i] = make_int4((int)v[4 * i], (int)v[4 * i + 1], (int)v[4 * i + 2], (int)v[4 * i + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (k < n) p[lay.at(row, t0 + k)] = (int32_t)v[k];
  }
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: the launches carry the programmatic stream
// serialization attribute, so a kernel may be scheduled while the previous
// kernel of the stream drains.  pdl_wait() blocks until that kernel has
// completed and its writes are visible (no-op when launched without the
// attribute); it comes before the first global access.  pdl_trigger() lets
// the next kernel of the stream start launching once every CTA of this grid
// has issued it (or exited).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// launch geometry
// ---------------------------------------------------------------------------
enum : int { kModeFull = 0, kModeAggregate = 1 };

// Geometry handed to every scan kernel.
struct Geom {
  int64_t E;
  int T;
  int seg_len;  // steps per segment, a multiple of the tile (>= T when nseg == 1)
  int nseg;     // segments per row; > 1 selects the two-pass path
  int mode;     // kModeFull or kModeAggregate (first pass of the two-pass path)
  int vec;      // env-major only: 16-byte aligned rows, T % 4 == 0
  int early;    // inputs do not depend on the previous kernel of the stream: load
                // before waiting on it, wait only before the first global write
  void* ws;     // [E][nseg] affine maps of the segments (two-pass path)
};

// consecutive steps per thread in the env-major driver (a multiple of 4:
// every 4 steps are one 16-byte vector of each float input)
#ifndef RLCA_EM_STEPS
#define RLCA_EM_STEPS 4
#endif
constexpr int kEmSteps = RLCA_EM_STEPS;

// env-major: TPR threads per row, kEmSteps steps per thread, rows packed 256 threads per CTA
template <int TPR>
struct EmShape {
  static constexpr int L = kEmSteps;
  static constexpr int TILE = TPR * L;
  static constexpr int BLOCK = TPR >= 256 ? TPR : 256;
  static constexpr int ROWS = BLOCK / TPR;
  static constexpr int GW = TPR < 32 ? TPR : 32;       // lanes of one row inside a warp
  static constexpr int NWR = TPR > 32 ? TPR / 32 : 1;  // warps per row
};

// time-major: 32 environments per warp, C chunk-threads per environment, L steps each
template <int C>
struct TmShape {
  static constexpr int L = 8;
  static constexpr int EW = 32;
  static constexpr int BLOCK = EW * C;
  static constexpr int TILE = C * L;
};

// value at a segment's far edge: the row's carry pushed through the maps of
// the segments between it and the row's end (written by the first pass of
// the two-pass path)
template <class V, bool BWD>
__device__ __forceinline__ V segment_carry_in(const Geom& g, int64_t row, int seg, V row_carry) {
  V c = row_carry;
  const Aff<V>* ws = reinterpret_cast<const Aff<V>*>(g.ws) + row * g.nseg;
  if (BWD) {
    for (int s = g.nseg - 1; s > seg; --s) c = ws[s].a + ws[s].b * c;
  } else {
    for (int s = 0; s < seg; ++s) c = ws[s].a + ws[s].b * c;
  }
  return c;
}

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

    est.template stage<S::ROWS, S::BLOCK, S::TILE>(lay, row0, rloc, ts, te, est_smem);
    typename Est::template Regs<L> R;
    est.template load<L>(R, lay, row, rloc, t0, n, vec, ts, S::TILE, S::ROWS, est_smem);
    if (it == ntiles - 1) pdl_trigger();

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
      if (n > 0 && edge && tn >= 0 && tn < g.T) est.nb_load(lay, row, tn, got);
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
      Aff<V>* x = xw + ((it & 1) * S::ROWS + rloc) * NWR;
      if (lane == (BWD ? 0 : 31)) x[wr] = inc;
      __syncthreads();
      Aff<V> cc = carry;
      boundary = cc;
      if (BWD) {
#pragma unroll 4
        for (int w = NWR - 1; w >= 0; --w) {
          if (w == wr) boundary = cc;
          cc = compose(x[w], cc);
        }
      } else {
#pragma unroll 4
        for (int w = 0; w < NWR; ++w) {
          if (w == wr) boundary = cc;
          cc = compose(x[w], cc);
        }
      }
      next_carry = cc;
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
      est.template store<L>(R, lay, row, t0, n, vec);
    }
    carry = next_carry;
  }
  if (agg_mode && row_ok && j == 0) reinterpret_cast<Aff<V>*>(g.ws)[row * g.nseg + seg] = carry;
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

    est.template stage_tm<S::BLOCK>(lay, row0, ts, te, est_smem);
    typename Est::template Regs<L> R;
    est.template load<L>(R, lay, row, lane, t0, n, false, ts, S::TILE, 32, est_smem);
    if (it == ntiles - 1) pdl_trigger();
    if constexpr (Est::kNb > 0) {
      float got[Est::kNb > 0 ? Est::kNb : 1];
#pragma unroll
      for (int i = 0; i < Est::kNb; ++i) got[i] = 0.f;
      const int tn = BWD ? t0 + L : t0 - 1;
      if (n > 0 && tn >= 0 && tn < g.T) est.nb_load(lay, row, tn, got);
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
      est.template store<L>(R, lay, row, t0, n, false);
    }
    carry = cc;
  }
  if (agg_mode && row_ok && cw == 0) reinterpret_cast<Aff<V>*>(g.ws)[row * g.nseg + seg] = carry;
}

}  // namespace rlca
