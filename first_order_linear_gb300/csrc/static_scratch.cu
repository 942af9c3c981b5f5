// static_scratch.cu -- rlca_gae_static_scratch: GAE without a caller workspace.
//
// Some callers cannot allocate device memory for the two-pass path's
// workspace (a C host that links only this library, a simulator callback that
// must not touch the device heap, a process that reserved all device memory
// up front).  For them the scratch lives in one file-scope device array of
// RLCA_STATIC_SCRATCH_BYTES that every GPU loading the library holds until
// exit.  Host code only sees a stand-in for that array's name, so its device
// address is looked up once per device context (with that device current)
// and handed to the kernel like any workspace.  Nothing here allocates.
#include <cuda.h>  // CUcontext / CUresult types of the two driver calls below

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "rlca.h"

namespace {

constexpr int kMaxDevices = 256;

static __device__ __align__(256) unsigned char g_gae_scratch[RLCA_STATIC_SCRATCH_BYTES];

std::atomic<int> g_sms[kMaxDevices];

// The array's address belongs to the device context the module was loaded
// into: after cudaDeviceReset (or any teardown of the primary context) the
// module is loaded again and the array may sit elsewhere.  Each cached
// address is therefore stored with the unique id of its context and looked
// up again when the current context's id differs.  The driver's
// cuCtxGetCurrent and cuCtxGetId are reached through the runtime's entry
// point query, so the library still links only the runtime.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxApi {
  CtxGetCurrentFn current = nullptr;
  CtxGetIdFn id = nullptr;
};

const CtxApi& ctx_api() {
  static const CtxApi api = [] {
    CtxApi a;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      a.id = reinterpret_cast<CtxGetIdFn>(f);
    return a;
  }();
  return api;
}

// unique id of the context current on this thread; 0 when there is none or
// it cannot be told (then the address is looked up on every call)
unsigned long long current_context_id() {
  const CtxApi& a = ctx_api();
  if (a.current == nullptr || a.id == nullptr) return 0;
  CUcontext c = nullptr;
  if (a.current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return a.id(c, &id) == CUDA_SUCCESS ? id : 0;
}

struct ScratchSlot {
  std::mutex m;
  unsigned long long ctx = 0;  // context the address was looked up in
  void* addr = nullptr;
};
ScratchSlot g_slot[kMaxDevices];

// set-up: device address of g_gae_scratch on the current device, looked up
// on a device's first call and again whenever its context has changed
cudaError_t scratch_address(int dev, void** out) {
  ScratchSlot& s = g_slot[dev];
  std::lock_guard<std::mutex> lock(s.m);
  const unsigned long long id = current_context_id();
  if (s.addr != nullptr && id != 0 && id == s.ctx) {
    *out = s.addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_gae_scratch);  // makes the device's context current
  if (e != cudaSuccess) return e;
  s.addr = p;
  s.ctx = current_context_id();
  *out = p;
  return cudaSuccess;
}

cudaError_t sm_count(int dev, int* out) {
  int c = g_sms[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_sms[dev].store(c, std::memory_order_relaxed);
  }
  *out = c;
  return cudaSuccess;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (a == nullptr || b == nullptr) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned(const void* p, uintptr_t a) { return p == nullptr || ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" int rlca_gae_static_scratch(const float* rewards, const float* values, const uint8_t* terminated,
                                       const uint8_t* truncated, const float* trunc_value, const float* bootstrap,
                                       float* advantages, float* returns, int64_t E, int64_t T, float gamma,
                                       float lambda, uint32_t flags, rlca_stream_t stream) {
  using namespace rlca;
  if (E < 0 || T < 0 || E > INT32_MAX || T > (int64_t(1) << 30)) return RLCA_ERR_INVALID_ARG;
  if (E == 0 || T == 0) return RLCA_OK;
  if (flags & RLCA_BF16) return RLCA_ERR_UNSUPPORTED;
  if ((flags & ~(RLCA_TIME_MAJOR | RLCA_MULTIPASS)) != 0u) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !values || !advantages || (truncated && !trunc_value)) return RLCA_ERR_INVALID_ARG;
  const size_t nf = (size_t)(E * T) * 4, nb = (size_t)(E * T);
  const void* ins[6] = {rewards, values, terminated, truncated, trunc_value, bootstrap};
  const size_t in_bytes[6] = {nf, nf, nb, nb, nf, (size_t)E * 4};
  for (int i = 0; i < 6; ++i)
    if (overlaps(advantages, nf, ins[i], in_bytes[i]) || overlaps(returns, nf, ins[i], in_bytes[i]))
      return RLCA_ERR_INVALID_ARG;
  if (overlaps(advantages, nf, returns, nf)) return RLCA_ERR_INVALID_ARG;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RLCA_ERR_CUDA;
  int sms = 0;
  if (sm_count(dev, &sms) != cudaSuccess) return RLCA_ERR_CUDA;
  const bool vec = aligned(rewards, 16) && aligned(values, 16) && aligned(advantages, 16) && aligned(returns, 16) &&
                   aligned(terminated, 4) && aligned(truncated, 4);
  Plan p;
  if (!make_plan(Kind::Gae, E, (int)T, 0, flags, sms, vec && T % 4 == 0, &p)) return RLCA_ERR_INVALID_ARG;
  if (p.ws_bytes > RLCA_STATIC_SCRATCH_BYTES) return RLCA_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (p.ws_bytes > 0 && scratch_address(dev, &ws) != cudaSuccess) return RLCA_ERR_CUDA;

  Geom g;
  g.E = E;
  g.T = (int)T;
  g.seg_len = p.seg_len;
  g.nseg = p.nseg;
  g.mode = kModeFull;
  g.vec = (!p.time_major && vec && T % 4 == 0) ? 1 : 0;
  g.early = 0;
  g.ws = ws;
  g.aux = nullptr;
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  cudaError_t e;
  if (truncated) {
    GaeEst<true> est;
    est.b = b; est.r = rewards; est.v = values; est.adv = advantages; est.ret = returns;
    est.gamma = gamma; est.gl = gamma * lambda;
    e = run_scan(est, p, g, stream);
  } else {
    GaeEst<false> est;
    est.b = b; est.r = rewards; est.v = values; est.adv = advantages; est.ret = returns;
    est.gamma = gamma; est.gl = gamma * lambda;
    e = run_scan(est, p, g, stream);
  }
  if (e != cudaSuccess) return RLCA_ERR_CUDA;
  return checked_build_status(stream);
}
