// estimators.cuh -- per-estimator coefficient construction for the scan drivers.
//
// Each functor turns raw rollout inputs into the (alpha_t, beta_t) of the
// recurrence in registers, as rl-triton (arXiv:2608.17641) §3.1 describes
// (fused kernels build the coefficients on chip from the raw rollout
// tensors), with the episode-boundary rules of §3.2:
//   termination  -> successor value 0, beta_t = 0
//   truncation   -> successor value trunc_value[t], beta_t = 0
//                   (termination wins where both flags are set)
//   t = T-1      -> successor value bootstrap, either inside alpha_{T-1}
//                   (GAE, V-Trace, Retrace; beta_{T-1} = 0) or through the
//                   scan carry A_T = bootstrap (TD(lambda), discounted return)
//   forward scans restart after a flagged step (§5: beta_t = 0 when d_{t-1} = 1).
//
// Interface used by the drivers of scan_core.cuh:
//   V, kBackward, kNb           value type, scan direction, neighbour floats
//   Regs<L>                     per-thread registers of L consecutive steps
//   row_carry(row)              A_T (backward) / A_{-1} (forward) of a row
//   stage / stage_tm            cooperative per-tile staging (Retrace only)
//   load(R, io, ...)            read the thread's L steps through io (io.cuh)
//   nb_give / nb_load / nb_take the neighbour step's inputs (step t0+L for a
//                               backward scan, t0-1 for a forward one)
//   coef(R, k, t)               (alpha_t, beta_t) of step t = t0 + k
//   emit(R, k, A, adj, c)       output of step k from A_t (adj = A of the
//                               step the recurrence reads)
//   store(R, io)                write the thread's outputs through io
//   kStageable, staged_io(f)    inputs the staged driver may stage (floats,
//                               then flag bytes)
#pragma once

#include <type_traits>

#include "io.cuh"

namespace rlca {

// Default no-op staging.
struct NoStage {
  template <int ROWS, int BLOCK, int TILE, class Lay>
  __device__ __forceinline__ void stage(const Lay&, const Geom&, int64_t, int, int, int, unsigned char*) const {}
  template <int BLOCK, class Lay>
  __device__ __forceinline__ void stage_tm(const Lay&, const Geom&, int64_t, int, int, unsigned char*) const {}
};

// Common boundary inputs of the backward estimators.
struct BoundaryArgs {
  const uint8_t* term;   // nullable
  const uint8_t* trunc;  // nullable (HAS_TRUNC == false ignores it)
  const float* tv;       // read where trunc is set
  const float* boot;     // [E], nullable
  int T;
};

template <int L>
struct BoundaryRegs {
  uint32_t term, trunc;  // bit k: flag of step t0+k (trunc already cleared where term is set)
  float tv[L];
  float boot;            // bootstrap of the row when this thread holds step T-1
};

// flags are staged byte inputs 0 (terminated) and 1 (truncated)
template <bool HAS_TRUNC, class ST, int L, class IO>
__device__ __forceinline__ void load_boundary(const BoundaryArgs& b, BoundaryRegs<L>& R, const IO& io) {
  R.term = io.template flags<L>(0, b.term);
  R.trunc = HAS_TRUNC ? (io.template flags<L>(1, b.trunc) & ~R.term) : 0u;
#pragma unroll
  for (int k = 0; k < L; ++k) R.tv[k] = 0.f;
  if (HAS_TRUNC && R.trunc != 0u) {  // truncations are rare: one branch instead of L predicated loads
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (((R.trunc >> k) & 1u) && in_range(io.at(k), io.total())) R.tv[k] = Stor<ST>::ld(b.tv, io.at(k));
  }
  R.boot = (io.n > 0 && io.t0 + io.n == b.T && b.boot != nullptr && in_range(io.row, io.envs()))
               ? Stor<ST>::ld(b.boot, io.row)
               : 0.f;
}

template <class F>
__host__ __device__ __forceinline__ void staged_flags(const BoundaryArgs& b, F& f) {
  f.in_b(b.term);
  f.in_b(b.trunc);
}

// successor value of step k: 0 / trunc value / bootstrap / interior value
template <int L>
__device__ __forceinline__ float successor(const BoundaryRegs<L>& R, int k, int t, int T, float interior) {
  float s = (t == T - 1) ? R.boot : interior;
  if ((R.trunc >> k) & 1u) s = R.tv[k];
  if ((R.term >> k) & 1u) s = 0.f;
  return s;
}

template <int L>
__device__ __forceinline__ bool cut(const BoundaryRegs<L>& R, int k) {
  return ((R.term | R.trunc) >> k) & 1u;
}

// ===========================================================================
// GAE (rl-triton §2.1; Schulman et al. 2016)
//   alpha_t = delta_t = r_t + gamma V_next(t) - V_t
//   beta_t  = gamma lambda (1 - d_t) [t < T-1],    carry 0
//   outputs adv_t = A_t, ret_t = A_t + V_t
// ===========================================================================
template <bool HAS_TRUNC, class ST = float>
struct GaeEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 2, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(r);
    f.in_f(v);
    staged_flags(b, f);
  }
  BoundaryArgs b;
  const float* r;
  const float* v;
  float* adv;
  float* ret;  // nullable
  float gamma, gl;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], v[L], vnext;
    float oa[L], orr[L];
  };
  __device__ __forceinline__ float row_carry(int64_t) const { return 0.f; }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, r, R.r);
    io.template f<L>(1, v, R.v);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
    R.vnext = 0.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const { g[0] = R.v[0]; }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = Stor<ST>::ld(v, lay.at(row, t));
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.vnext = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const float vn = successor(R.bd, k, t, b.T, (k + 1 < L) ? R.v[k + 1] : R.vnext);
    const float delta = R.r[k] + gamma * vn - R.v[k];
    const float beta = (cut(R.bd, k) || t == b.T - 1) ? 0.f : gl;
    return {delta, beta};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.oa[k] = A;
    R.orr[k] = A + R.v[k];
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, adv, R.oa);
    io.template put<L>(1, ret, R.orr);
  }
};

// ===========================================================================
// Discounted return
//   alpha_t = r_t + gamma trunc_t trunc_value_t,  beta_t = gamma (1 - d_t),
//   carry A_T = bootstrap
// ===========================================================================
template <bool HAS_TRUNC, class ST = float>
struct DiscEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 0;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 1, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(r);
    staged_flags(b, f);
  }
  BoundaryArgs b;
  const float* r;
  float* out;
  float gamma;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], o[L];
  };
  __device__ __forceinline__ float row_carry(int64_t row) const {
    return b.boot != nullptr ? Stor<ST>::ld(b.boot, row) : 0.f;
  }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, r, R.r);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>&, float*) const {}
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay&, int64_t, int, float*) const {}
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>&, const float*) const {}
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int) const {
    const bool tr = (R.bd.trunc >> k) & 1u;
    const float alpha = tr ? R.r[k] + gamma * R.bd.tv[k] : R.r[k];
    return {alpha, cut(R.bd, k) ? 0.f : gamma};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

// ===========================================================================
// TD(lambda) return
//   alpha_t = r_t + gamma [trunc_t tv_t + (1 - d_t)(1 - lambda) V_next(t)]
//   beta_t  = gamma lambda (1 - d_t),   carry A_T = bootstrap
// ===========================================================================
template <bool HAS_TRUNC, class ST = float>
struct TdLambdaEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 2, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(r);
    f.in_f(v);
    staged_flags(b, f);
  }
  BoundaryArgs b;
  const float* r;
  const float* v;
  float* out;
  float gamma, gl, one_minus_lambda;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], v[L], vnext, o[L];
  };
  __device__ __forceinline__ float row_carry(int64_t row) const {
    return b.boot != nullptr ? Stor<ST>::ld(b.boot, row) : 0.f;
  }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, r, R.r);
    io.template f<L>(1, v, R.v);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
    R.vnext = 0.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const { g[0] = R.v[0]; }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = Stor<ST>::ld(v, lay.at(row, t));
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.vnext = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const bool tm = (R.bd.term >> k) & 1u, tr = (R.bd.trunc >> k) & 1u;
    const float vn = (t == b.T - 1) ? R.bd.boot : ((k + 1 < L) ? R.v[k + 1] : R.vnext);
    const float tail = tm ? 0.f : (tr ? R.bd.tv[k] : one_minus_lambda * vn);
    return {R.r[k] + gamma * tail, (tm || tr) ? 0.f : gl};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

// ===========================================================================
// Fused value targets: GAE (adv, ret), discounted return and TD(lambda) of
// one rollout from a single read of r, V and the flags.  GAE and the
// discounted return are the recurrences of GaeEst and DiscEst, scanned side
// by side as one F2-valued affine map per step (.x GAE, .y discounted
// return; carry A_T = (0, bootstrap)).  The TD(lambda) return is written as
// adv + V: the lambda-return satisfies G_t = A_t + V_t exactly under every
// boundary rule (interior: r + gamma[(1-lambda)V_{t+1} + lambda G_{t+1}];
// termination: r; truncation: r + gamma tv; window edge: r + gamma b), so
// it needs no third scan.
// ===========================================================================
template <bool HAS_TRUNC, class ST = float>
struct ValueTargetsEst : NoStage {
  using Store = ST;
  using V = F2;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 2, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(r);
    f.in_f(v);
    staged_flags(b, f);
  }
  BoundaryArgs b;
  const float* r;
  const float* v;
  float* adv;   // each output nullable
  float* ret;
  float* disc;
  float* td;
  float gamma, gl;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], v[L], vnext;
    float oa[L], od[L];
  };
  __device__ __forceinline__ F2 row_carry(int64_t row) const {
    return F2(0.f, b.boot != nullptr ? Stor<ST>::ld(b.boot, row) : 0.f);
  }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, r, R.r);
    io.template f<L>(1, v, R.v);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
    R.vnext = 0.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const { g[0] = R.v[0]; }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = Stor<ST>::ld(v, lay.at(row, t));
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.vnext = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<F2> coef(const Regs<L>& R, int k, int t) const {
    const bool tr = (R.bd.trunc >> k) & 1u;
    const bool c = cut(R.bd, k);
    const float vn = successor(R.bd, k, t, b.T, (k + 1 < L) ? R.v[k + 1] : R.vnext);
    const float delta = R.r[k] + gamma * vn - R.v[k];
    const float a_disc = tr ? R.r[k] + gamma * R.bd.tv[k] : R.r[k];
    return {F2(delta, a_disc), F2((c || t == b.T - 1) ? 0.f : gl, c ? 0.f : gamma)};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, F2 A, F2, const Aff<F2>&) const {
    R.oa[k] = A.x;
    R.od[k] = A.y;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    float ret_[L];
#pragma unroll
    for (int k = 0; k < L; ++k) ret_[k] = R.oa[k] + R.v[k];
    io.template put<L>(0, adv, R.oa);
    io.template put<L>(1, ret, ret_);
    io.template put<L>(2, disc, R.od);
    io.template put<L>(3, td, ret_);
  }
};

// ===========================================================================
// V-Trace (rl-triton §8; Espeholt et al. 2018)
//   rho_t = min(rho_bar, ratio_t),  c_t = lambda min(c_bar, ratio_t)
//   alpha_t = rho_t (r_t + gamma V_next(t) - V_t)
//   beta_t  = gamma c_t (1 - d_t) [t < T-1],   carry 0
//   vs_t = V_t + A_t;  pg_t = rho_t (r_t + gamma vs_next(t) - V_t)
// ===========================================================================
template <bool HAS_TRUNC, class ST = float>
struct VtraceEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 4, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(r);
    f.in_f(v);
    f.in_f(lpt);
    f.in_f(lpb);
    staged_flags(b, f);
  }
  BoundaryArgs b;
  const float* r;
  const float* v;
  const float* lpt;
  const float* lpb;
  float* vs;
  float* pg;  // nullable
  float gamma, rho_bar, c_bar, lambda;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], v[L], rho[L], c[L], vnext;
    float ovs[L], opg[L];
    int t0;
  };
  __device__ __forceinline__ float row_carry(int64_t) const { return 0.f; }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    float a[L], bb[L];
    io.template f<L>(0, r, R.r);
    io.template f<L>(1, v, R.v);
    io.template f<L>(2, lpt, a);
    io.template f<L>(3, lpb, bb);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
#pragma unroll
    for (int k = 0; k < L; ++k) {
      // the hardware exponential: a relative error of a few ulp, far inside
      // the 1e-4 tolerance, at a fraction of the accurate expf's instructions
      const float ratio = __expf(a[k] - bb[k]);
      R.rho[k] = fminf(rho_bar, ratio);
      R.c[k] = lambda * fminf(c_bar, ratio);
    }
    R.vnext = 0.f;
    R.t0 = io.t0;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const { g[0] = R.v[0]; }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = Stor<ST>::ld(v, lay.at(row, t));
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.vnext = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const float vn = successor(R.bd, k, t, b.T, (k + 1 < L) ? R.v[k + 1] : R.vnext);
    const float delta = R.rho[k] * (R.r[k] + gamma * vn - R.v[k]);
    const float beta = (cut(R.bd, k) || t == b.T - 1) ? 0.f : gamma * R.c[k];
    return {delta, beta};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float adj, const Aff<float>&) const {
    R.ovs[k] = R.v[k] + A;
    const float vn = (k + 1 < L) ? R.v[k + 1] : R.vnext;
    const float nvs = successor(R.bd, k, R.t0 + k, b.T, vn + adj);
    R.opg[k] = R.rho[k] * (R.r[k] + gamma * nvs - R.v[k]);
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, vs, R.ovs);
    io.template put<L>(1, pg, R.opg);
  }
};

// ===========================================================================
// Retrace(lambda) (rl-triton §3.3; Munos et al. 2016)
//   per step (reduced over the action axis on chip, before the scan):
//     EV_t = sum_a pi[t,a] Q[t,a],  Qa_t = Q[t,a_t],  c_t = lambda min(1, pi[t,a_t] / mu_a[t])
//   alpha_t = r_t + gamma (EV_{t+1} - c_{t+1} Qa_{t+1})   inside an episode
//           = r_t (termination) / r_t + gamma tv_t (truncation) / r_t + gamma bootstrap (t = T-1)
//   beta_t  = gamma c_{t+1} (1 - d_t) [t < T-1],   carry 0
// The per-step reduction stages the [items, A] blocks of Q and pi through
// shared memory with coalesced loads; each tile stages its steps plus the
// first step after it (the last step's successor).
// ===========================================================================
// per-warp raw Q / pi buffers of the Retrace staging: 1 = one 32-step chunk
// at a time, 2 = the next chunk's copies in flight while this one reduces.
// Env-major rows keep one (more CTAs resident measured faster); time-major
// tiles, with few CTAs of up to 8 warps, take two.
__host__ __device__ constexpr int retrace_bufs(bool time_major) { return time_major ? 2 : 1; }
// floats of shared memory per warp for the raw blocks: buffers x (Q, pi) x 32 steps x A
__host__ __device__ constexpr int retrace_raw_floats(int A, bool time_major) {
  return retrace_bufs(time_major) * 64 * A;
}

template <class ST = float>
struct RetraceStage {
  static constexpr int ES = (int)sizeof(ST);  // bytes of a stored element
  using Bits = typename std::conditional<ES == 2, unsigned short, uint32_t>::type;
  const float* q;     // [.., A] elements of type ST
  const float* pi;    // [.., A] elements of type ST
  const float* mu_a;  // elements of type ST
  const int32_t* act;
  int A;
  float lambda;
  int64_t items;  // E * T steps (read by the index-check build)

  struct Pending {
    int at;
    float mu;
  };
  // bytes [b0, nbytes) of a block into shared memory: 16-byte asynchronous
  // pieces while both sources allow them, then 4-byte pieces, then (an
  // unaligned block, or the last half word of a bfloat16 one) plain loads
  __device__ __forceinline__ static void copy_block(unsigned char* dq, unsigned char* dp, const unsigned char* qb,
                                                    const unsigned char* pb, int nbytes, int lane) {
    int b0 = 0;
    const uintptr_t al = reinterpret_cast<uintptr_t>(qb) | reinterpret_cast<uintptr_t>(pb);
    if ((al & 15u) == 0) {
      const int n16 = nbytes >> 4;
      for (int f = lane; f < n16; f += 32) {
        cp_async16(dq + 16 * f, qb + 16 * f);
        cp_async16(dp + 16 * f, pb + 16 * f);
      }
      b0 = 16 * n16;
    }
    if ((al & 3u) == 0) {
      const int n4 = nbytes >> 2;
      for (int f = (b0 >> 2) + lane; f < n4; f += 32) {
        cp_async4(dq + 4 * f, qb + 4 * f);
        cp_async4(dp + 4 * f, pb + 4 * f);
      }
      b0 = 4 * n4;
    }
    for (int f = b0 / ES + lane; f < nbytes / ES; f += 32) {
      reinterpret_cast<Bits*>(dq)[f] = __ldg(reinterpret_cast<const Bits*>(qb) + f);
      reinterpret_cast<Bits*>(dp)[f] = __ldg(reinterpret_cast<const Bits*>(pb) + f);
    }
  }
  // items e0 .. e0+cnt-1 (element indices of [.., A] rows, contiguous): the
  // warp's Q and pi blocks go to shared memory, the copies all in flight at
  // once and committed as one group (the shared buffers start on 16-byte
  // boundaries); the taken action and mu(a_t) load into registers alongside
  __device__ __forceinline__ Pending issue(int64_t e0, int cnt, int lane, float* raw_q, float* raw_p) const {
    if (!span_in_range(e0, cnt, items)) cnt = 0;  // index-check build: skip the block
    const unsigned char* qb = reinterpret_cast<const unsigned char*>(q) + e0 * A * ES;
    const unsigned char* pb = reinterpret_cast<const unsigned char*>(pi) + e0 * A * ES;
    copy_block(reinterpret_cast<unsigned char*>(raw_q), reinterpret_cast<unsigned char*>(raw_p), qb, pb,
               cnt * A * ES, lane);
    cp_async_commit();
    Pending pd;
    pd.at = lane < cnt ? __ldg(act + e0 + lane) : 0;
    pd.mu = lane < cnt ? Stor<ST>::ld(mu_a, e0 + lane) : 1.f;
    return pd;
  }
  __device__ __forceinline__ static float elem(const float* raw, int i) {
    if constexpr (ES == 4) {
      return raw[i];
    } else {
      return __uint_as_float((uint32_t)reinterpret_cast<const Bits*>(raw)[i] << 16);
    }
  }
  // once the chunk's copies have landed: item `lane` writes its three
  // scalars at index `slot` of the dst arrays
  __device__ __forceinline__ void finish(const Pending& pd, int cnt, int lane, const float* raw_q,
                                         const float* raw_p, float* dst_ev, float* dst_qa, float* dst_c,
                                         int slot, int nslots) const {
    if (lane < cnt && in_range(slot, nslots)) {
      const int base = lane * A;
      float ev = 0.f;
      if constexpr (ES == 4) {
        const float* rq = raw_q + base;
        const float* rp = raw_p + base;
        if ((A & 1) == 0) {  // 8-byte aligned pairs, same summation order
          const float2* q2 = reinterpret_cast<const float2*>(rq);
          const float2* p2 = reinterpret_cast<const float2*>(rp);
          for (int a = 0; a < A / 2; ++a) {
            const float2 x = q2[a], y = p2[a];
            ev = fmaf(y.x, x.x, ev);
            ev = fmaf(y.y, x.y, ev);
          }
        } else {
          for (int a = 0; a < A; ++a) ev = fmaf(rp[a], rq[a], ev);
        }
      } else if ((A & 1) == 0) {  // 4-byte aligned pairs of bfloat16, same summation order
        const uint32_t* q2 = reinterpret_cast<const uint32_t*>(raw_q) + base / 2;
        const uint32_t* p2 = reinterpret_cast<const uint32_t*>(raw_p) + base / 2;
        for (int a = 0; a < A / 2; ++a) {
          const uint32_t x = q2[a], y = p2[a];
          ev = fmaf(__uint_as_float(y << 16), __uint_as_float(x << 16), ev);
          ev = fmaf(__uint_as_float(y & 0xffff0000u), __uint_as_float(x & 0xffff0000u), ev);
        }
      } else {
        for (int a = 0; a < A; ++a) ev = fmaf(elem(raw_p, base + a), elem(raw_q, base + a), ev);
      }
      const int at = pd.at < 0 ? 0 : (pd.at >= A ? A - 1 : pd.at);
      dst_ev[slot] = ev;
      dst_qa[slot] = elem(raw_q, base + at);
      dst_c[slot] = lambda * fminf(1.f, elem(raw_p, base + at) / pd.mu);
    }
  }
  // walks chunks warp, warp + NW, ... < nch; where(ch, &e0, &cnt, &slot)
  // locates a chunk (false: nothing to stage).  With two buffers the next
  // chunk's copies are issued before waiting on the current one.
  template <int NBUF, class Where>
  __device__ __forceinline__ void walk(int nch, int warp, int NW, int lane, float* raw, float* s_ev, float* s_qa,
                                       float* s_c, int nslots, Where where) const {
    const int blk = 32 * A;
    auto buf = [&](int k) { return raw + (NBUF == 2 ? (k & 1) : 0) * 2 * blk; };
    int64_t e0 = 0;
    int cnt = 0, slot = 0;
    Pending cur = {0, 1.f};
    bool cur_ok = false;
    if (NBUF == 2 && warp < nch) {
      cur_ok = where(warp, &e0, &cnt, &slot);
      if (cur_ok) cur = issue(e0, cnt, lane, buf(0), buf(0) + blk);
    }
    int k = 0;
    for (int ch = warp; ch < nch; ch += NW, ++k) {
      if (NBUF == 2) {
        const int nx = ch + NW;
        int64_t ne0 = 0;
        int ncnt = 0, nslot = 0;
        const bool nx_ok = nx < nch && where(nx, &ne0, &ncnt, &nslot);
        Pending nxt = {0, 1.f};
        if (nx_ok) {
          nxt = issue(ne0, ncnt, lane, buf(k + 1), buf(k + 1) + blk);
          cp_async_wait<1>();
        } else {
          cp_async_wait<0>();
        }
        __syncwarp();
        if (cur_ok) finish(cur, cnt, lane, buf(k), buf(k) + blk, s_ev, s_qa, s_c, slot, nslots);
        __syncwarp();
        cur = nxt;
        cur_ok = nx_ok;
        e0 = ne0;
        cnt = ncnt;
        slot = nslot;
      } else {
        if (!where(ch, &e0, &cnt, &slot)) continue;
        const Pending pd = issue(e0, cnt, lane, raw, raw + blk);
        cp_async_wait<0>();
        __syncwarp();
        finish(pd, cnt, lane, raw, raw + blk, s_ev, s_qa, s_c, slot, nslots);
        __syncwarp();
      }
    }
  }
};

template <bool HAS_TRUNC, class ST = float>
struct RetraceEst {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 0;
  static constexpr bool kStageable = false;
  static constexpr int kSF = 0, kSB = 0;  // staged float inputs, flag inputs
  BoundaryArgs b;
  RetraceStage<ST> st;
  const float* r;
  float* out;
  float gamma;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], evn[L], qan[L], cn[L], o[L];
  };
  __device__ __forceinline__ float row_carry(int64_t) const { return 0.f; }

  // shared memory: per warp the raw Q and pi blocks (retrace_raw_floats),
  // then the staged per-step scalars [3][ROWS][tile + 1].  On the two-pass
  // path (g.aux set) the first pass also copies each tile's own steps'
  // scalars to the planes g.aux, and the second pass fills the staged
  // scalars from there instead of reading Q and pi again.
  template <int ROWS, int BLOCK, int TILE, class Lay>
  __device__ __forceinline__ void stage(const Lay& lay, const Geom& g, int64_t row0, int, int ts, int te,
                                        unsigned char* sm) const {
    constexpr int NW = BLOCK / 32;
    constexpr int SROW = TILE + 1;  // tile + 1 steps per row
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* raw = reinterpret_cast<float*>(sm) + warp * retrace_raw_floats(st.A, false);
    float* s_ev = reinterpret_cast<float*>(sm) + NW * retrace_raw_floats(st.A, false);
    float* s_qa = s_ev + ROWS * SROW;
    float* s_c = s_qa + ROWS * SROW;
    const int nst = te - ts + (te < b.T ? 1 : 0);
    const int64_t plane = lay.E * (int64_t)lay.T;
    if (g.aux != nullptr && g.mode == kModeFull) {
      // every load of the tile in flight at once, then the shared-memory writes
      constexpr int PER = (ROWS * SROW + BLOCK - 1) / BLOCK;
      float ev[PER], qa[PER], cc[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = threadIdx.x + u * BLOCK;
        const int rr = i / nst, k = i - rr * nst;
        const bool ok = i < ROWS * nst && row0 + rr < lay.E && in_range(lay.at(row0 + rr, ts + k), plane);
        const int64_t gi = ok ? lay.at(row0 + rr, ts + k) : 0;
        ev[u] = ok ? __ldg(g.aux + gi) : 0.f;
        qa[u] = ok ? __ldg(g.aux + plane + gi) : 0.f;
        cc[u] = ok ? __ldg(g.aux + 2 * plane + gi) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = threadIdx.x + u * BLOCK;
        const int rr = i / nst, k = i - rr * nst;
        if (i < ROWS * nst && row0 + rr < lay.E) {
          s_ev[rr * SROW + k] = ev[u];
          s_qa[rr * SROW + k] = qa[u];
          s_c[rr * SROW + k] = cc[u];
        }
      }
      __syncthreads();
      return;
    }
    const int per_row = (nst + 31) / 32;
    st.template walk<retrace_bufs(false)>(ROWS * per_row, warp, NW, lane, raw, s_ev, s_qa, s_c, ROWS * SROW,
            [&](int ch, int64_t* e0, int* cnt, int* slot) {
              const int rr = ch / per_row, m = ch - rr * per_row;
              if (row0 + rr >= lay.E) return false;
              const int i0 = m * 32;
              *e0 = lay.at(row0 + rr, ts + i0);
              *cnt = min(32, nst - i0);
              *slot = rr * SROW + i0 + lane;
              return true;
            });
    __syncthreads();
    if (g.aux != nullptr) {  // first pass: steps ts .. te-1 are this tile's own
      const int own = te - ts;
      for (int i = threadIdx.x; i < ROWS * own; i += BLOCK) {
        const int rr = i / own, k = i - rr * own;
        if (row0 + rr < lay.E && in_range(lay.at(row0 + rr, ts + k), plane)) {
          const int64_t gi = lay.at(row0 + rr, ts + k);
          g.aux[gi] = s_ev[rr * SROW + k];
          g.aux[plane + gi] = s_qa[rr * SROW + k];
          g.aux[2 * plane + gi] = s_c[rr * SROW + k];
        }
      }
    }
  }
  // time-major: one chunk = one step of 32 consecutive environments;
  // staged scalars [3][tile + 1][32]; the planes as in stage()
  template <int BLOCK, class Lay>
  __device__ __forceinline__ void stage_tm(const Lay& lay, const Geom& g, int64_t row0, int ts, int te,
                                           unsigned char* sm) const {
    constexpr int NW = BLOCK / 32;
    constexpr int SROWS = (BLOCK / 32) * 8 + 1;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* raw = reinterpret_cast<float*>(sm) + warp * retrace_raw_floats(st.A, true);
    float* s_ev = reinterpret_cast<float*>(sm) + NW * retrace_raw_floats(st.A, true);
    float* s_qa = s_ev + SROWS * 32;
    float* s_c = s_qa + SROWS * 32;
    const int nst = te - ts + (te < b.T ? 1 : 0);
    const int cnt = (int)min((int64_t)32, lay.E - row0);
    const int64_t plane = lay.E * (int64_t)lay.T;
    if (g.aux != nullptr && g.mode == kModeFull) {
      // every load of the tile in flight at once, then the shared-memory
      // writes (one round trip instead of one per loop pass)
      constexpr int PER = (SROWS * 32 + BLOCK - 1) / BLOCK;
      float ev[PER], qa[PER], cc[PER];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = threadIdx.x + u * BLOCK;
        const int k = i >> 5, l = i & 31;
        const bool ok = i < nst * 32 && l < cnt && in_range(lay.at(row0 + l, ts + k), plane) &&
                        in_range(i, SROWS * 32);
        const int64_t gi = ok ? lay.at(row0 + l, ts + k) : 0;
        ev[u] = ok ? __ldg(g.aux + gi) : 0.f;
        qa[u] = ok ? __ldg(g.aux + plane + gi) : 0.f;
        cc[u] = ok ? __ldg(g.aux + 2 * plane + gi) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int i = threadIdx.x + u * BLOCK;
        if (i < nst * 32 && i < SROWS * 32) {
          s_ev[i] = ev[u];
          s_qa[i] = qa[u];
          s_c[i] = cc[u];
        }
      }
      __syncthreads();
      return;
    }
    st.template walk<retrace_bufs(true)>(nst, warp, NW, lane, raw, s_ev, s_qa, s_c, SROWS * 32, [&](int i, int64_t* e0, int* c, int* slot) {
      *e0 = lay.at(row0, ts + i);
      *c = cnt;
      *slot = i * 32 + lane;
      return true;
    });
    __syncthreads();
    if (g.aux != nullptr) {  // first pass: steps ts .. te-1 are this tile's own
      for (int i = threadIdx.x; i < (te - ts) * 32; i += BLOCK) {
        const int k = i >> 5, l = i & 31;
        if (l < cnt && in_range(lay.at(row0 + l, ts + k), plane) && in_range(i, SROWS * 32)) {
          const int64_t gi = lay.at(row0 + l, ts + k);
          g.aux[gi] = s_ev[i];
          g.aux[plane + gi] = s_qa[i];
          g.aux[2 * plane + gi] = s_c[i];
        }
      }
    }
  }

  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int slot, int ts, int tile, int nrows,
                                       unsigned char* sm) const {
    io.template f<L>(0, r, R.r);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
    constexpr bool kTM = IO::kTimeMajor;
    const int t0 = io.t0, n = io.n;
    const int NW = blockDim.x >> 5;
    const float* s_ev = reinterpret_cast<const float*>(sm) + NW * retrace_raw_floats(st.A, kTM);
    const int srows = tile + 1;
    const int plane = srows * nrows;
    const float* s_qa = s_ev + plane;
    const float* s_c = s_qa + plane;
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const int t = t0 + k + 1;  // successor step
      const int i = t - ts;
      const int idx = kTM ? i * 32 + slot : slot * srows + i;
      if (k < n && t < b.T && in_range(idx, plane)) {
        R.evn[k] = s_ev[idx];
        R.qan[k] = s_qa[idx];
        R.cn[k] = s_c[idx];
      } else {
        R.evn[k] = 0.f;
        R.qan[k] = 0.f;
        R.cn[k] = 0.f;
      }
    }
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>&, float*) const {}
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay&, int64_t, int, float*) const {}
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>&, const float*) const {}
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const bool tm = (R.bd.term >> k) & 1u, tr = (R.bd.trunc >> k) & 1u;
    const bool last = t == b.T - 1;
    const float interior = R.evn[k] - R.cn[k] * R.qan[k];
    const float tail = tm ? 0.f : (tr ? R.bd.tv[k] : (last ? R.bd.boot : interior));
    const float beta = (tm || tr || last) ? 0.f : gamma * R.cn[k];
    return {R.r[k] + gamma * tail, beta};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

// Second pass of Retrace's two-pass split.  The first pass left every
// step's (EV, Qa, c) in three float planes of the workspace (element order
// of the inputs), so this pass is a scan of scalars: r, the flags and the
// successor step's three plane values build the same (alpha_t, beta_t) as
// RetraceEst::coef, without the per-action blocks or shared-memory staging.
// It runs on the fast time-major driver, whose CTAs of 8 (16 for bfloat16)
// environments give the few-environment, long-row problems that take the
// split several times the CTAs of the first pass.
template <bool HAS_TRUNC, class ST = float>
struct RetraceTailEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = true;
  static constexpr int kNb = 3;  // the next chunk's first (EV, Qa, c)
  static constexpr bool kStageable = false;
  static constexpr int kSF = 0, kSB = 0;
  BoundaryArgs b;
  const float* r;
  const float* aux;  // planes EV, Qa, c of E * T floats each
  int64_t plane;     // E * T
  float* out;
  float gamma;

  template <int L>
  struct Regs {
    BoundaryRegs<L> bd;
    float r[L], ev[L], qa[L], c[L], o[L];
    float evn, qan, cn;  // step t0 + L
  };
  __device__ __forceinline__ float row_carry(int64_t) const { return 0.f; }

  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, r, R.r);
    load_boundary<HAS_TRUNC, ST, L>(b, R.bd, io);
#pragma unroll
    for (int k = 0; k < L; ++k) {
      const int64_t i = io.at(k);
      const bool ok = k < io.n && in_range(i, plane);
      R.ev[k] = ok ? __ldg(aux + i) : 0.f;
      R.qa[k] = ok ? __ldg(aux + plane + i) : 0.f;
      R.c[k] = ok ? __ldg(aux + 2 * plane + i) : 0.f;
    }
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const {
    g[0] = R.ev[0];
    g[1] = R.qa[0];
    g[2] = R.c[0];
  }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    const int64_t i = lay.at(row, t);
    g[0] = __ldg(aux + i);
    g[1] = __ldg(aux + plane + i);
    g[2] = __ldg(aux + 2 * plane + i);
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const {
    R.evn = g[0];
    R.qan = g[1];
    R.cn = g[2];
  }
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const float evs = k + 1 < L ? R.ev[k + 1] : R.evn;
    const float qas = k + 1 < L ? R.qa[k + 1] : R.qan;
    const float cs = k + 1 < L ? R.c[k + 1] : R.cn;
    const bool tm = (R.bd.term >> k) & 1u, tr = (R.bd.trunc >> k) & 1u;
    const bool last = t == b.T - 1;
    const float interior = evs - cs * qas;
    const float tail = tm ? 0.f : (tr ? R.bd.tv[k] : (last ? R.bd.boot : interior));
    const float beta = (tm || tr || last) ? 0.f : gamma * cs;
    return {R.r[k] + gamma * tail, beta};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

// ===========================================================================
// Eligibility trace, forward (rl-triton §1, §5)
//   alpha_t = x_t,  beta_t = gamma lambda (1 - d_{t-1}),  e_{-1} = 0
// ===========================================================================
template <class ST = float>
struct EligEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = false;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 1, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(x);
    f.in_b(term);
    f.in_b(trunc);
  }
  const float* x;
  const uint8_t* term;   // nullable
  const uint8_t* trunc;  // nullable
  float* out;
  float gl;

  template <int L>
  struct Regs {
    float x[L], o[L];
    uint32_t done;
    float prev_done;
  };
  __device__ __forceinline__ float row_carry(int64_t) const { return 0.f; }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, x, R.x);
    R.done = io.template flags<L>(0, term) | io.template flags<L>(1, trunc);
    R.prev_done = 1.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const {
    g[0] = ((R.done >> (L - 1)) & 1u) ? 1.f : 0.f;
  }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = (load_flag1(term, lay, row, t) || load_flag1(trunc, lay, row, t)) ? 1.f : 0.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.prev_done = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int t) const {
    const bool start = (t == 0) || (k == 0 ? R.prev_done != 0.f : ((R.done >> (k - 1)) & 1u) != 0u);
    return {R.x[k], start ? 0.f : gl};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

// ===========================================================================
// Episodic prefix sum, segmented forward scan (rl-triton §3.3)
//   alpha_t = x_t,  beta_t = 1 - start_t, where start_t = d_{t-1} (flag ends
//   an episode) or d_t (flag starts one), and start_0 = 1.
//   exclusive output: beta_t * A_{t-1}.
// int32 runs in uint32 arithmetic (wraps modulo 2^32; beta is 0 or 1, so any
// grouping gives the same bits).
// ===========================================================================
template <class VT, class ST = float>
struct PrefixSumEst : NoStage {
  using Store = ST;
  using V = VT;
  static constexpr bool kBackward = false;
  static constexpr int kNb = 1;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 1, kSB = 2;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(x);
    f.in_b(term);
    f.in_b(trunc);
  }
  const void* x;
  const uint8_t* term;
  const uint8_t* trunc;
  void* out;
  int exclusive;
  int flag_is_start;

  template <int L>
  struct Regs {
    V x[L], o[L];
    uint32_t done;
    float prev_done;
  };
  __device__ __forceinline__ V row_carry(int64_t) const { return V(0); }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    if constexpr (std::is_integral<V>::value) {
      io.template i<L>(0, static_cast<const int32_t*>(x), R.x);
    } else {
      io.template f<L>(0, static_cast<const float*>(x), R.x);
    }
    R.done = io.template flags<L>(0, term) | io.template flags<L>(1, trunc);
    R.prev_done = 1.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>& R, float* g) const {
    g[0] = ((R.done >> (L - 1)) & 1u) ? 1.f : 0.f;
  }
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay& lay, int64_t row, int t, float* g) const {
    g[0] = (load_flag1(term, lay, row, t) || load_flag1(trunc, lay, row, t)) ? 1.f : 0.f;
  }
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>& R, const float* g) const { R.prev_done = g[0]; }
  template <int L>
  __device__ __forceinline__ Aff<V> coef(const Regs<L>& R, int k, int t) const {
    bool start;
    if (flag_is_start)
      start = (t == 0) || ((R.done >> k) & 1u);
    else
      start = (t == 0) || (k == 0 ? R.prev_done != 0.f : ((R.done >> (k - 1)) & 1u) != 0u);
    return {R.x[k], start ? V(0) : V(1)};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, V A, V adj, const Aff<V>& c) const {
    R.o[k] = exclusive ? (c.b != V(0) ? adj : V(0)) : A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    if constexpr (std::is_integral<V>::value) {
      io.template put_i<L>(0, static_cast<int32_t*>(out), R.o);
    } else {
      io.template put<L>(0, static_cast<float*>(out), R.o);
    }
  }
};

// ===========================================================================
// Generic affine scan over precomputed coefficients (rl-triton §4)
// ===========================================================================
template <bool BWD, class ST = float>
struct AffineEst : NoStage {
  using Store = ST;
  using V = float;
  static constexpr bool kBackward = BWD;
  static constexpr int kNb = 0;
  static constexpr bool kStageable = true;
  static constexpr int kSF = 2, kSB = 0;  // staged float inputs, flag inputs
  template <class F>
  __host__ __device__ __forceinline__ void staged_io(F& f) const {
    f.in_f(alpha);
    f.in_f(beta);
  }
  const float* alpha;
  const float* beta;
  const float* carry;  // [E], nullable
  float* out;

  template <int L>
  struct Regs {
    float a[L], b[L], o[L];
  };
  __device__ __forceinline__ float row_carry(int64_t row) const {
    return carry != nullptr ? Stor<ST>::ld(carry, row) : 0.f;
  }
  template <int L, class IO>
  __device__ __forceinline__ void load(Regs<L>& R, const IO& io, int, int, int, int, unsigned char*) const {
    io.template f<L>(0, alpha, R.a);
    io.template f<L>(1, beta, R.b);
  }
  template <int L>
  __device__ __forceinline__ void nb_give(const Regs<L>&, float*) const {}
  template <class Lay>
  __device__ __forceinline__ void nb_load(const Lay&, int64_t, int, float*) const {}
  template <int L>
  __device__ __forceinline__ void nb_take(Regs<L>&, const float*) const {}
  template <int L>
  __device__ __forceinline__ Aff<float> coef(const Regs<L>& R, int k, int) const {
    return {R.a[k], R.b[k]};
  }
  template <int L>
  __device__ __forceinline__ void emit(Regs<L>& R, int k, float A, float, const Aff<float>&) const {
    R.o[k] = A;
  }
  template <int L, class IO>
  __device__ __forceinline__ void store(const Regs<L>& R, const IO& io) const {
    io.template put<L>(0, out, R.o);
  }
};

}  // namespace rlca
