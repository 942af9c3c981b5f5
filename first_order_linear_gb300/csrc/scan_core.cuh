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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace rlca {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// device status word and the index-check build.  Each translation unit has
// its own word (internal linkage); the host reads them with
// rlca_device_status.  A kernel records a condition here instead of
// trapping: a bounded wait that gave up, or (built with RLCA_INDEX_CHECK) an
// index outside its array, whose access is then skipped or clamped.
// ---------------------------------------------------------------------------
static __device__ unsigned int g_tu_status;
constexpr unsigned int kStatusWaitTimeout = 1u;
constexpr unsigned int kStatusIndex = 2u;
#ifdef RLCA_INDEX_CHECK
constexpr bool kIndexCheck = true;
#else
constexpr bool kIndexCheck = false;
#endif
// 0 <= i < n; in the index-check build a miss is recorded (the caller skips
// the access); otherwise always true and free
__device__ __forceinline__ bool in_range(int64_t i, int64_t n) {
  if constexpr (kIndexCheck) {
    if (i < 0 || i >= n) {
      atomicOr(&g_tu_status, kStatusIndex);
      return false;
    }
  }
  return true;
}
// [i, i + len) inside [0, n)
__device__ __forceinline__ bool span_in_range(int64_t i, int64_t len, int64_t n) {
  if constexpr (kIndexCheck) return in_range(i, n) && in_range(i + len - 1, n);
  return true;
}

// ---------------------------------------------------------------------------
// storage of the floating-point arrays.  Arithmetic and the scan state are
// float32 always; with RLCA_BF16 every float array of a call holds bfloat16
// (the upper half of a float32), converted on load and rounded to nearest
// even once on store.  An estimator's float pointers then point at elements
// of type ST; Stor<ST> does the element access.
// ---------------------------------------------------------------------------
using bf16 = __nv_bfloat16;

template <class ST>
struct Stor;

template <>
struct Stor<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float ld(const float* p, int64_t i) { return __ldg(p + i); }
  __device__ __forceinline__ static void st(float* p, int64_t i, float v) { p[i] = v; }
  // four consecutive elements starting at a 16-byte boundary (zeros where !ok)
  __device__ __forceinline__ static void ld4(const float* p, int64_t i, bool ok, float* o) {
    const float4 v = ok ? __ldg(reinterpret_cast<const float4*>(p + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    o[0] = v.x, o[1] = v.y, o[2] = v.z, o[3] = v.w;
  }
  __device__ __forceinline__ static void st4(float* p, int64_t i, const float* v) {
    *reinterpret_cast<float4*>(p + i) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

template <>
struct Stor<bf16> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float from_bits(uint32_t h) { return __uint_as_float(h << 16); }
  __device__ __forceinline__ static uint32_t to_bits(float v) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  __device__ __forceinline__ static float ld(const float* p, int64_t i) {
    return from_bits(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
  }
  __device__ __forceinline__ static void st(float* p, int64_t i, float v) {
    reinterpret_cast<unsigned short*>(p)[i] = (unsigned short)to_bits(v);
  }
  // four consecutive elements starting at an 8-byte boundary (zeros where !ok)
  __device__ __forceinline__ static void ld4(const float* p, int64_t i, bool ok, float* o) {
    const uint2 w =
        ok ? __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(p) + i)) : make_uint2(0, 0);
    o[0] = __uint_as_float(w.x << 16), o[1] = __uint_as_float(w.x & 0xffff0000u);
    o[2] = __uint_as_float(w.y << 16), o[3] = __uint_as_float(w.y & 0xffff0000u);
  }
  // two elements rounded to nearest even in one conversion, the first in
  // the low half (the element at the lower address)
  __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ static void st4(float* p, int64_t i, const float* v) {
    const uint2 w = make_uint2(pack2(v[0], v[1]), pack2(v[2], v[3]));
    *reinterpret_cast<uint2*>(reinterpret_cast<unsigned short*>(p) + i) = w;
  }
  // eight consecutive elements starting at a 16-byte boundary (zeros where !ok)
  __device__ __forceinline__ static void ld8(const float* p, int64_t i, bool ok, float* o) {
    const uint4 w =
        ok ? __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p) + i)) : make_uint4(0, 0, 0, 0);
    o[0] = __uint_as_float(w.x << 16), o[1] = __uint_as_float(w.x & 0xffff0000u);
    o[2] = __uint_as_float(w.y << 16), o[3] = __uint_as_float(w.y & 0xffff0000u);
    o[4] = __uint_as_float(w.z << 16), o[5] = __uint_as_float(w.z & 0xffff0000u);
    o[6] = __uint_as_float(w.w << 16), o[7] = __uint_as_float(w.w & 0xffff0000u);
  }
  __device__ __forceinline__ static void st8(float* p, int64_t i, const float* v) {
    const uint4 w = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned short*>(p) + i) = w;
  }
};

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

// Two independent recurrences scanned side by side (the fused value-target
// scan: GAE and the discounted return of one row).  Arithmetic is
// element-wise, so compose() on Aff<F2> composes both maps at once.
struct F2 {
  float x, y;
  F2() = default;
  __host__ __device__ constexpr F2(float s) : x(s), y(s) {}
  __host__ __device__ constexpr F2(float a, float b) : x(a), y(b) {}
};
__device__ __forceinline__ F2 operator+(const F2& a, const F2& b) { return {a.x + b.x, a.y + b.y}; }
__device__ __forceinline__ F2 operator*(const F2& a, const F2& b) { return {a.x * b.x, a.y * b.y}; }

__device__ __forceinline__ float shfl_down_v(float v, int d, int w) { return __shfl_down_sync(kFullMask, v, d, w); }
__device__ __forceinline__ uint32_t shfl_down_v(uint32_t v, int d, int w) {
  return __shfl_down_sync(kFullMask, v, d, w);
}
__device__ __forceinline__ F2 shfl_down_v(const F2& v, int d, int w) {
  return {shfl_down_v(v.x, d, w), shfl_down_v(v.y, d, w)};
}
__device__ __forceinline__ float shfl_up_v(float v, int d, int w) { return __shfl_up_sync(kFullMask, v, d, w); }
__device__ __forceinline__ uint32_t shfl_up_v(uint32_t v, int d, int w) { return __shfl_up_sync(kFullMask, v, d, w); }
__device__ __forceinline__ F2 shfl_up_v(const F2& v, int d, int w) {
  return {shfl_up_v(v.x, d, w), shfl_up_v(v.y, d, w)};
}
__device__ __forceinline__ float shfl_idx_v(float v, int s, int w) { return __shfl_sync(kFullMask, v, s, w); }
__device__ __forceinline__ uint32_t shfl_idx_v(uint32_t v, int s, int w) { return __shfl_sync(kFullMask, v, s, w); }
__device__ __forceinline__ F2 shfl_idx_v(const F2& v, int s, int w) {
  return {shfl_idx_v(v.x, s, w), shfl_idx_v(v.y, s, w)};
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
template <int L, class Lay, class ST = float>
__device__ __forceinline__ void load_vals(const float* __restrict__ p, const Lay& lay, int64_t row,
                                          int t0, int n, bool vec, float (&out)[L]) {
  const int64_t tot = lay.E * (int64_t)lay.T;
  if (vec) {
    const int64_t base = lay.at(row, t0);
    if constexpr (sizeof(ST) == 2 && L % 8 == 0) {  // 16-byte vectors of 8 bfloat16 steps
#pragma unroll
      for (int i = 0; i < L / 8; ++i)
        Stor<ST>::ld8(p, base + 8 * i, 8 * i < n && span_in_range(base + 8 * i, 8, tot), &out[8 * i]);
    } else {
#pragma unroll
      for (int i = 0; i < L / 4; ++i)
        Stor<ST>::ld4(p, base + 4 * i, 4 * i < n && span_in_range(base + 4 * i, 4, tot), &out[4 * i]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      out[k] = (k < n && in_range(lay.at(row, t0 + k), tot)) ? Stor<ST>::ld(p, lay.at(row, t0 + k)) : 0.f;
  }
}

template <int L, class Lay>
__device__ __forceinline__ void load_ints(const int32_t* __restrict__ p, const Lay& lay, int64_t row,
                                          int t0, int n, bool vec, uint32_t (&out)[L]) {
  const int64_t tot = lay.E * (int64_t)lay.T;
  if (vec) {
    const int4* q = reinterpret_cast<const int4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i) {
      int4 v = (4 * i < n && span_in_range(lay.at(row, t0) + 4 * i, 4, tot)) ? __ldg(q + i) : make_int4(0, 0, 0, 0);
      out[4 * i + 0] = (uint32_t)v.x;
      out[4 * i + 1] = (uint32_t)v.y;
      out[4 * i + 2] = (uint32_t)v.z;
      out[4 * i + 3] = (uint32_t)v.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      out[k] = (k < n && in_range(lay.at(row, t0 + k), tot)) ? (uint32_t)__ldg(p + lay.at(row, t0 + k)) : 0u;
  }
}

// bit k of the result = (flag at step t0+k != 0); 0 for a NULL array
template <int L, class Lay>
__device__ __forceinline__ uint32_t load_flags(const uint8_t* __restrict__ p, const Lay& lay, int64_t row,
                                               int t0, int n, bool vec) {
  if (p == nullptr) return 0u;
  uint32_t bits = 0u;
  const int64_t tot = lay.E * (int64_t)lay.T;
  if (vec) {
    const uint32_t* q = reinterpret_cast<const uint32_t*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i) {
      const uint32_t w = (4 * i < n && span_in_range(lay.at(row, t0) + 4 * i, 4, tot)) ? __ldg(q + i) : 0u;
      // one bit per nonzero byte: bytes -> 0/1, then the multiply gathers
      // byte k's bit into bit 24 + k (the partial products never overlap)
      const uint32_t m = __vcmpne4(w, 0u) & 0x01010101u;
      bits |= ((m * 0x01020408u) >> 24) << (4 * i);
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k) {
      if (k < n && in_range(lay.at(row, t0 + k), tot) && __ldg(p + lay.at(row, t0 + k)) != 0) bits |= 1u << k;
    }
  }
  return bits;
}

template <class Lay>
__device__ __forceinline__ bool load_flag1(const uint8_t* __restrict__ p, const Lay& lay, int64_t row, int t) {
  return p != nullptr && in_range(lay.at(row, t), lay.E * (int64_t)lay.T) && __ldg(p + lay.at(row, t)) != 0;
}

template <int L, class Lay, class ST = float>
__device__ __forceinline__ void store_vals(float* __restrict__ p, const Lay& lay, int64_t row, int t0,
                                           int n, bool vec, const float (&v)[L]) {
  const int64_t tot = lay.E * (int64_t)lay.T;
  if (vec) {
    const int64_t base = lay.at(row, t0);
    if constexpr (sizeof(ST) == 2 && L % 8 == 0) {
#pragma unroll
      for (int i = 0; i < L / 8; ++i)
        if (8 * i < n && span_in_range(base + 8 * i, 8, tot)) Stor<ST>::st8(p, base + 8 * i, &v[8 * i]);
    } else {
#pragma unroll
      for (int i = 0; i < L / 4; ++i)
        if (4 * i < n && span_in_range(base + 4 * i, 4, tot)) Stor<ST>::st4(p, base + 4 * i, &v[4 * i]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (k < n && in_range(lay.at(row, t0 + k), tot)) Stor<ST>::st(p, lay.at(row, t0 + k), v[k]);
  }
}

template <int L, class Lay>
__device__ __forceinline__ void store_ints(int32_t* __restrict__ p, const Lay& lay, int64_t row, int t0,
                                           int n, bool vec, const uint32_t (&v)[L]) {
  const int64_t tot = lay.E * (int64_t)lay.T;
  if (vec) {
    int4* q = reinterpret_cast<int4*>(p + lay.at(row, t0));
#pragma unroll
    for (int i = 0; i < L / 4; ++i)
      if (4 * i < n && span_in_range(lay.at(row, t0) + 4 * i, 4, tot))
        q[i] = make_int4((int)v[4 * i], (int)v[4 * i + 1], (int)v[4 * i + 2], (int)v[4 * i + 3]);
  } else {
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (k < n && in_range(lay.at(row, t0 + k), tot)) p[lay.at(row, t0 + k)] = (int32_t)v[k];
  }
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: the launches carry the programmatic stream
// serialization attribute, so a kernel may be scheduled while the previous
// kernel of the stream drains.  pdl_wait() blocks until that kernel has
// completed and its writes are visible (no-op when launched without the
// attribute); it comes before the first global access that may conflict
// with it.  pdl_trigger() lets the next kernel of the stream start
// launching once every CTA of this grid has issued it (or exited).  It
// carries no memory ordering -- the next kernel's own pdl_wait() still
// waits for this grid's completion -- so every driver issues it first
// thing: the next launch's CTAs then take free SM slots (and, with
// RLCA_INPUTS_READY, load their inputs) while this grid still runs.
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
  float* aux;   // Retrace, two-pass path: per-step (E_pi Q, Q(a_t), c_t) as three
                // planes of E * T floats in the call's element order (else null)
};

// consecutive steps per thread in the env-major driver (a multiple of 4:
// every 4 steps are one 16-byte vector of each float input)
#ifndef RLCA_EM_STEPS
#define RLCA_EM_STEPS 4
#endif
constexpr int kEmSteps = RLCA_EM_STEPS;

// rows of at least this many steps use 8 steps per thread in the fast
// driver (half the warps per row)
#ifndef RLCA_FAST_L8_MIN_T
#define RLCA_FAST_L8_MIN_T 1024
#endif
constexpr int kFastL8MinT = RLCA_FAST_L8_MIN_T;

// smallest env-major CTA (rows shorter than this share a CTA)
#ifndef RLCA_EM_MIN_BLOCK
#define RLCA_EM_MIN_BLOCK 128
#endif
constexpr int kEmMinBlock = RLCA_EM_MIN_BLOCK;

// env-major: TPR threads per row, kEmSteps steps per thread, rows packed kEmMinBlock threads per CTA
template <int TPR, int LS = kEmSteps>
struct EmShape {
  static constexpr int L = LS;
  static constexpr int TILE = TPR * L;
  static constexpr int BLOCK = TPR >= kEmMinBlock ? TPR : kEmMinBlock;
  static constexpr int ROWS = BLOCK / TPR;
  static constexpr int GW = TPR < 32 ? TPR : 32;       // lanes of one row inside a warp
  static constexpr int NWR = TPR > 32 ? TPR / 32 : 1;  // warps per row
};

__host__ __device__ constexpr size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// async global -> shared copies (completed by cp_async_wait_all, a hardware
// wait on the thread's own copies)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// waits until at most N of this thread's committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// time-major: 32 environments per warp, C chunk-threads per environment, L steps each
template <int C>
struct TmShape {
  static constexpr int L = 8;
  static constexpr int EW = 32;
  static constexpr int BLOCK = EW * C;
  static constexpr int TILE = C * L;
};

// fast time-major: EW environments per CTA (EW consecutive floats of a step
// row per load), CT chunk-threads per environment, L steps each.  Thread tid
// loads and emits environment tid % EW, chunk tid / EW; for the scan across
// chunks it takes environment tid / CT, chunk tid % CT, so an environment's
// CT chunk maps sit in CT adjacent lanes of one warp.
template <int EW, int CT>
struct TfShape {
  static constexpr int L = 8;
  static constexpr int BLOCK = EW * CT;
  static constexpr int TILE = CT * L;
  static constexpr int PAD = EW + 1;  // row stride of the [CT][EW] exchange arrays
  static_assert(BLOCK % 32 == 0 && CT <= 32 && (CT & (CT - 1)) == 0, "chunk groups tile the warps");
};
// resident CTAs the fast time-major drivers are compiled for: 32 warps per
// SM for CTAs of 128 threads or more, i.e. at most 64 registers a thread (a
// few more cost a whole CTA); tiny CTAs (T < 32) are left unbounded
__host__ __device__ constexpr int tf_min_blocks(int block) {
  return block >= 1024 ? 1 : (1024 / block < 8 ? 1024 / block : 8);
}
template <class V, int EW, int CT>
__host__ __device__ constexpr size_t tf_smem_bytes() {
  return (size_t)CT * TfShape<EW, CT>::PAD * (sizeof(Aff<V>) + sizeof(V));
}

// staged time-major: the fast time-major shape with its inputs copied into
// a ring of NS shared-memory stages, one tile per stage.  In a stage each
// staged input is a [CT][CS] buffer: chunk c's step k, environment j at
// c * CS + k * EW + j.  CS pads a chunk by EW elements when several chunks
// share a warp (EW < 32), so their lanes read distinct banks.
#ifndef RLCA_TS_STAGES
#define RLCA_TS_STAGES 2
#endif
template <int EW, int CT>
struct TsShape : TfShape<EW, CT> {
  static constexpr int NS = RLCA_TS_STAGES;
  static constexpr int CS = TfShape<EW, CT>::L * EW + (EW < 32 ? EW : 0);
  static constexpr int FB = CT * CS;  // elements per staged buffer
  static_assert(EW % 4 == 0 && CS % 4 == 0, "16-byte pieces of step rows");
};
template <class Est, int EW, int CT>
__host__ __device__ constexpr size_t ts_stage_bytes() {
  return align16((size_t)TsShape<EW, CT>::FB * (sizeof(typename Est::Store) * Est::kSF + Est::kSB));
}
template <class Est, int EW, int CT>
__host__ __device__ constexpr size_t ts_smem_bytes() {
  return align16(tf_smem_bytes<typename Est::V, EW, CT>()) + TsShape<EW, CT>::NS * ts_stage_bytes<Est, EW, CT>();
}

// value at a segment's far edge: the row's carry pushed through the maps of
// the segments between it and the row's end (written by the first pass of
// the two-pass path)
template <class V, bool BWD>
__device__ __forceinline__ V segment_carry_in(const Geom& g, int64_t row, int seg, V row_carry) {
  V c = row_carry;
  const Aff<V>* ws = reinterpret_cast<const Aff<V>*>(g.ws) + row * g.nseg;
  const int64_t nmaps = g.E * (int64_t)g.nseg;
  if (BWD) {
    for (int s = g.nseg - 1; s > seg; --s)
      if (in_range(row * g.nseg + s, nmaps)) c = ws[s].a + ws[s].b * c;
  } else {
    for (int s = 0; s < seg; ++s)
      if (in_range(row * g.nseg + s, nmaps)) c = ws[s].a + ws[s].b * c;
  }
  return c;
}

}  // namespace rlca
