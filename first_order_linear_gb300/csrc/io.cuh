// io.cuh -- where an estimator's per-thread inputs come from and its outputs go.
//
// Estimator functors read their L consecutive steps and write their outputs
// through an I/O object, so the same functor serves
//   GIO: global memory (the direct env-major and time-major drivers), and
//   SIO: shared memory staged by the CTA with coalesced async copies (the
//        staged env-major driver; see staged.cuh).
// Inputs are addressed by (index, pointer): the index is the position in the
// estimator's staged_io() list and is what SIO uses; GIO uses the pointer.
#pragma once

#include "scan_core.cuh"

namespace rlca {

// VEC_CT: the vector path is known at compile time (fast driver); otherwise
// `vec` decides at run time
template <class Lay, bool VEC_CT = false>
struct GIO {
  static constexpr bool kTimeMajor = Lay::kTimeMajor;
  const Lay& lay;
  int64_t row;
  int t0;
  int n;
  bool vec_rt;
  __device__ __forceinline__ bool vec() const { return VEC_CT || vec_rt; }

  __device__ __forceinline__ int64_t at(int k) const { return lay.at(row, t0 + k); }
  template <int L>
  __device__ __forceinline__ void f(int, const float* p, float (&o)[L]) const {
    load_vals<L>(p, lay, row, t0, n, vec(), o);
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
    if (p != nullptr) store_vals<L>(p, lay, row, t0, n, vec(), v);
  }
  template <int L>
  __device__ __forceinline__ void put_i(int, int32_t* p, const uint32_t (&v)[L]) const {
    if (p != nullptr) store_ints<L>(p, lay, row, t0, n, vec(), v);
  }
};

// Shared-memory staging layout of one CTA tile (env-major, SL steps per
// thread): float buffer b holds thread slot s's SL values at
// b * fstride + s * (SL + 4) (the 4-float pad makes the per-thread 16-byte
// reads and writes of a quarter warp hit distinct banks); byte buffer b holds
// slot s's SL flags at b * bstride + s * SL.  Outputs reuse the float
// buffers after every thread has read its inputs.
template <int SL>
struct SIO {
  static constexpr bool kTimeMajor = false;
  static constexpr int kPad = SL + 4;
  float* fbuf;
  const uint8_t* bbuf;
  int fstride;
  int bstride;
  int slot;
  const EnvMajor& lay;
  int64_t row;
  int t0;
  int n;

  __device__ __forceinline__ int64_t at(int k) const { return lay.at(row, t0 + k); }
  template <int L>
  __device__ __forceinline__ void f(int idx, const float*, float (&o)[L]) const {
    static_assert(L == SL, "staged I/O serves SL steps per thread");
    const float4* s = reinterpret_cast<const float4*>(fbuf + idx * fstride + slot * kPad);
#pragma unroll
    for (int j = 0; j < L / 4; ++j) {
      const float4 v = s[j];
      o[4 * j] = v.x;
      o[4 * j + 1] = v.y;
      o[4 * j + 2] = v.z;
      o[4 * j + 3] = v.w;
    }
  }
  template <int L>
  __device__ __forceinline__ void i(int idx, const int32_t*, uint32_t (&o)[L]) const {
    const uint4* s = reinterpret_cast<const uint4*>(fbuf + idx * fstride + slot * kPad);
#pragma unroll
    for (int j = 0; j < L / 4; ++j) {
      const uint4 v = s[j];
      o[4 * j] = v.x;
      o[4 * j + 1] = v.y;
      o[4 * j + 2] = v.z;
      o[4 * j + 3] = v.w;
    }
  }
  template <int L>
  __device__ __forceinline__ uint32_t flags(int idx, const uint8_t* p) const {
    if (p == nullptr) return 0u;
    uint32_t w[L / 4];
    const unsigned char* src = bbuf + idx * bstride + slot * SL;
    if constexpr (L == 16) {
      const uint4 q = *reinterpret_cast<const uint4*>(src);
      w[0] = q.x, w[1] = q.y, w[2] = q.z, w[3] = q.w;
    } else if constexpr (L == 8) {
      const uint2 q = *reinterpret_cast<const uint2*>(src);
      w[0] = q.x, w[1] = q.y;
    } else {
#pragma unroll
      for (int j = 0; j < L / 4; ++j) w[j] = reinterpret_cast<const uint32_t*>(src)[j];
    }
    uint32_t bits = 0u;
#pragma unroll
    for (int j = 0; j < L / 4; ++j) {
      const uint32_t m = __vcmpne4(w[j], 0u) & 0x01010101u;
      bits |= ((m * 0x01020408u) >> 24) << (4 * j);
    }
    return bits;
  }
  template <int L>
  __device__ __forceinline__ void put(int idx, float* p, const float (&v)[L]) const {
    if (p == nullptr) return;
    float4* d = reinterpret_cast<float4*>(fbuf + idx * fstride + slot * kPad);
#pragma unroll
    for (int j = 0; j < L / 4; ++j) d[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
  template <int L>
  __device__ __forceinline__ void put_i(int idx, int32_t* p, const uint32_t (&v)[L]) const {
    if (p == nullptr) return;
    uint4* d = reinterpret_cast<uint4*>(fbuf + idx * fstride + slot * kPad);
#pragma unroll
    for (int j = 0; j < L / 4; ++j) d[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
};

// Collects an estimator's staged inputs and outputs (in staged_io order).
struct StagedList {
  static constexpr int kMaxF = 4, kMaxB = 2, kMaxO = 4;
  const void* fin[kMaxF];
  const uint8_t* bin[kMaxB];
  void* out[kMaxO];
  int nf = 0, nb = 0, no = 0;
  __device__ __forceinline__ void in_f(const void* p) { fin[nf++] = p; }
  __device__ __forceinline__ void in_b(const uint8_t* p) { bin[nb++] = p; }
  __device__ __forceinline__ void out_f(void* p) { out[no++] = p; }
};

}  // namespace rlca
