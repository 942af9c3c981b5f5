// io.cuh -- where an estimator's per-thread inputs come from and its outputs go.
//
// Estimator functors read their L consecutive steps and write their outputs
// through an I/O object, so the same functor serves
//   GIO: global memory (the direct env-major and time-major drivers),
//   TmIO32: global memory, time-major, 32-bit offsets (fast time-major driver),
//   TmSIO: shared-memory stages of the staged time-major driver.
// Inputs are addressed by (index, pointer): the index is the position in the
// estimator's staged_io() list and is what TmSIO uses; the global ones use
// the pointer.
#pragma once

#include "scan_core.cuh"

namespace rlca {

// VEC_CT: the vector path is known at compile time (fast driver); otherwise
// `vec` decides at run time.  ST: element type of the float arrays.
template <class Lay, bool VEC_CT = false, class ST = float>
struct GIO {
  static constexpr bool kTimeMajor = Lay::kTimeMajor;
  const Lay& lay;
  int64_t row;
  int t0;
  int n;
  bool vec_rt;
  __device__ __forceinline__ bool vec() const { return VEC_CT || vec_rt; }

  __device__ __forceinline__ int64_t at(int k) const { return lay.at(row, t0 + k); }
  __device__ __forceinline__ int64_t total() const { return lay.E * (int64_t)lay.T; }
  __device__ __forceinline__ int64_t envs() const { return lay.E; }
  template <int L>
  __device__ __forceinline__ void f(int, const float* p, float (&o)[L]) const {
    load_vals<L, Lay, ST>(p, lay, row, t0, n, vec(), o);
  }
  template <int L>
  __device__ __forceinline__ void i(int, const int32_t* p, uint32_t (&o)[L]) const {
    load_ints<L>(p, lay, row, t0, n, vec(), o);
  }
  template <int L>
  __device__ __forceinline__ uint32_t flags(int, const uint8_t* p) const {
    return load_flags<L>(p, lay, row, t0, n, vec());
  }
  template <int L>
  __device__ __forceinline__ void put(int, float* p, const float (&v)[L]) const {
    if (p != nullptr) store_vals<L, Lay, ST>(p, lay, row, t0, n, vec(), v);
  }
  template <int L>
  __device__ __forceinline__ void put_i(int, int32_t* p, const uint32_t (&v)[L]) const {
    if (p != nullptr) store_ints<L>(p, lay, row, t0, n, vec(), v);
  }
};

// Time-major [T, E] global I/O of the fast time-major driver: a thread's L
// steps are either all in range (n == L) or none (n == 0), and every array's
// element (t0 + k, row) sits at element offset off + k * E, computed in 32
// bits (the planner takes this path only when E * T < 2^32).
template <class ST = float>
struct TmIO32 {
  static constexpr bool kTimeMajor = true;
  int64_t row;
  int t0;
  int n;
  uint32_t off;  // t0 * E + row
  uint32_t E;
  uint32_t tot;  // E * T (read by the index-check build)

  __device__ __forceinline__ uint32_t o(int k) const { return off + (uint32_t)k * E; }
  __device__ __forceinline__ int64_t at(int k) const { return (int64_t)o(k); }
  __device__ __forceinline__ int64_t total() const { return tot; }
  __device__ __forceinline__ int64_t envs() const { return E; }
  template <int L>
  __device__ __forceinline__ void f(int, const float* __restrict__ p, float (&v)[L]) const {
#pragma unroll
    for (int k = 0; k < L; ++k) v[k] = (n != 0 && in_range(o(k), tot)) ? Stor<ST>::ld(p, o(k)) : 0.f;
  }
  template <int L>
  __device__ __forceinline__ void i(int, const int32_t* __restrict__ p, uint32_t (&v)[L]) const {
#pragma unroll
    for (int k = 0; k < L; ++k) v[k] = (n != 0 && in_range(o(k), tot)) ? (uint32_t)__ldg(p + o(k)) : 0u;
  }
  template <int L>
  __device__ __forceinline__ uint32_t flags(int, const uint8_t* __restrict__ p) const {
    if (p == nullptr || n == 0) return 0u;
    uint32_t bits = 0u;
#pragma unroll
    for (int k = 0; k < L; ++k) bits |= (uint32_t)(in_range(o(k), tot) && __ldg(p + o(k)) != 0) << k;
    return bits;
  }
  template <int L>
  __device__ __forceinline__ void put(int, float* __restrict__ p, const float (&v)[L]) const {
    if (p == nullptr || n == 0) return;
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (in_range(o(k), tot)) Stor<ST>::st(p, o(k), v[k]);
  }
  template <int L>
  __device__ __forceinline__ void put_i(int, int32_t* __restrict__ p, const uint32_t (&v)[L]) const {
    if (p == nullptr || n == 0) return;
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (in_range(o(k), tot)) p[o(k)] = (int32_t)v[k];
  }
};

// Time-major I/O of the staged time-major drivers: inputs from the current
// shared-memory stage (float input b at fbuf + b * FB elements of type ST,
// the thread's step k at slot + k * EW; flag input b at bbuf + b * FBB
// bytes, step k at fslot + k * FW: flag rows may be staged wider than the
// CTA's environments), outputs and the rare truncation-value loads straight
// to global memory as in TmIO32.
template <int EW, int FB, class ST = float, int FW = EW, int FBB = FB>
struct TmSIO {
  static constexpr bool kTimeMajor = true;
  const ST* fbuf;
  const uint8_t* bbuf;
  int slot;
  int fslot;
  int64_t row;
  int t0;
  int n;
  uint32_t off;  // t0 * E + row
  uint32_t E;
  uint32_t tot;  // E * T (read by the index-check build)

  __device__ __forceinline__ uint32_t o(int k) const { return off + (uint32_t)k * E; }
  __device__ __forceinline__ int64_t at(int k) const { return (int64_t)o(k); }
  __device__ __forceinline__ int64_t total() const { return tot; }
  __device__ __forceinline__ int64_t envs() const { return E; }
  template <int L>
  __device__ __forceinline__ void f(int idx, const float*, float (&v)[L]) const {
    const ST* s = fbuf + idx * FB + slot;
#pragma unroll
    for (int k = 0; k < L; ++k) v[k] = (n != 0 && in_range(slot + k * EW, FB)) ? static_cast<float>(s[k * EW]) : 0.f;
  }
  template <int L>
  __device__ __forceinline__ void i(int idx, const int32_t*, uint32_t (&v)[L]) const {
    static_assert(sizeof(ST) == 4, "int inputs are staged as 4-byte elements");
    const uint32_t* s = reinterpret_cast<const uint32_t*>(fbuf + idx * FB + slot);
#pragma unroll
    for (int k = 0; k < L; ++k) v[k] = (n != 0 && in_range(slot + k * EW, FB)) ? s[k * EW] : 0u;
  }
  template <int L>
  __device__ __forceinline__ uint32_t flags(int idx, const uint8_t* p) const {
    if (p == nullptr || n == 0) return 0u;
    const uint8_t* s = bbuf + idx * FBB + fslot;
    uint32_t bits = 0u;
#pragma unroll
    for (int k = 0; k < L; ++k) bits |= (uint32_t)(in_range(fslot + k * FW, FBB) && s[k * FW] != 0) << k;
    return bits;
  }
  template <int L>
  __device__ __forceinline__ void put(int, float* __restrict__ p, const float (&v)[L]) const {
    if (p == nullptr || n == 0) return;
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (in_range(o(k), tot)) Stor<ST>::st(p, o(k), v[k]);
  }
  template <int L>
  __device__ __forceinline__ void put_i(int, int32_t* __restrict__ p, const uint32_t (&v)[L]) const {
    if (p == nullptr || n == 0) return;
#pragma unroll
    for (int k = 0; k < L; ++k)
      if (in_range(o(k), tot)) p[o(k)] = (int32_t)v[k];
  }
};

// Collects an estimator's staged inputs (in staged_io order).
struct StagedList {
  static constexpr int kMaxF = 4, kMaxB = 2;
  const void* fin[kMaxF];
  const uint8_t* bin[kMaxB];
  int nf = 0, nb = 0;
  __host__ __device__ __forceinline__ void in_f(const void* p) { fin[nf++] = p; }
  __host__ __device__ __forceinline__ void in_b(const uint8_t* p) { bin[nb++] = p; }
};

}  // namespace rlca
