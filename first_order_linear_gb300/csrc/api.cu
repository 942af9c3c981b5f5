// api.cu -- the extern "C" entry points declared in include/rlca.h:
// argument validation on the host, launch planning, and launches on the
// caller's stream.  Nothing here allocates memory or synchronises.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <initializer_list>

#include "internal.h"
#include "rlca.h"

namespace rlca {

namespace {

constexpr int64_t kMaxT = int64_t(1) << 30;
constexpr int64_t kMaxE = INT32_MAX;
constexpr size_t kMaxMapBytes = sizeof(Aff<F2>);  // largest affine map of any estimator


int next_pow2(int64_t x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

std::atomic<int> g_sm_count[256];

cudaError_t sm_count_of_current_device(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 256) {
    int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return cudaSuccess;
    }
  }
  int c = 0;
  e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 256) g_sm_count[dev].store(c, std::memory_order_relaxed);
  *out = c;
  return cudaSuccess;
}

struct Span {
  const void* p;
  size_t bytes;
};

bool overlap(const Span& a, const Span& b) {
  if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
  const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// every output against every input and every other output
bool any_overlap(std::initializer_list<Span> ins, std::initializer_list<Span> outs) {
  for (const Span& o : outs) {
    for (const Span& i : ins)
      if (overlap(o, i)) return true;
    for (const Span& o2 : outs)
      if (&o2 != &o && overlap(o, o2)) return true;
  }
  return false;
}

bool aligned(const void* p, uintptr_t a) { return p == nullptr || ((uintptr_t)p % a) == 0; }

// sizes: negative / too large -> invalid; returns 1 when the call is decided
// (invalid, or empty and therefore done)
int check_sizes(int64_t E, int64_t T, int* status) {
  if (E < 0 || T < 0 || E > kMaxE || T > kMaxT) {
    *status = RLCA_ERR_INVALID_ARG;
    return 1;
  }
  if (E == 0 || T == 0) {
    *status = RLCA_OK;
    return 1;
  }
  return 0;
}

bool flags_ok(uint32_t flags, uint32_t allowed) { return (flags & ~allowed) == 0u; }

constexpr uint32_t kLayoutFlags = RLCA_TIME_MAJOR | RLCA_MULTIPASS | RLCA_INPUTS_READY;
// flags of the calls whose float arrays may be bfloat16
constexpr uint32_t kFloatFlags = kLayoutFlags | RLCA_BF16;

template <class T>
struct TypeTag {
  using type = T;
};
// f(TypeTag<ST>{}) with ST the element type of the call's float arrays
template <class F>
int with_storage(uint32_t flags, F&& f) {
  return (flags & RLCA_BF16) ? f(TypeTag<bf16>{}) : f(TypeTag<float>{});
}
// bytes of one float-array element
size_t fbytes(uint32_t flags) { return (flags & RLCA_BF16) ? 2 : 4; }

}  // namespace

// Index-check build (RLCA_INDEX_CHECK): every call waits for its kernels and
// fails with RLCA_ERR_CUDA when one of them recorded a condition in a device
// status word (the bits stay readable through rlca_device_status).  The
// product build returns RLCA_OK without waiting.
int checked_build_status(cudaStream_t s) {
  if constexpr (!kIndexCheck) {
    (void)s;
    return RLCA_OK;
  } else {
    if (cudaStreamSynchronize(s) != cudaSuccess) return RLCA_ERR_CUDA;
    unsigned int w = 0;
    if (rlca_device_status(&w, 0) != RLCA_OK) return RLCA_ERR_CUDA;
    return w == 0 ? RLCA_OK : RLCA_ERR_CUDA;
  }
}

namespace {

template <class Est>
int launch(Kind kind, const Est& est, int64_t E, int64_t T, int A, uint32_t flags, void* ws, size_t ws_bytes,
           bool vec_ok, cudaStream_t s) {
  int sm = 0;
  if (sm_count_of_current_device(&sm) != cudaSuccess) return RLCA_ERR_CUDA;
  // tensor-copy staging of time-major tiles: every staged input on a
  // 16-byte boundary (the copies' rule), E % 16 == 0 (16-byte flag rows)
  bool bulk = false;
  if constexpr (Est::kStageable) {
    if ((flags & RLCA_TIME_MAJOR) && E % 16 == 0 && tensor_maps_available()) {
      StagedList in;
      est.staged_io(in);
      bulk = true;
      for (int i = 0; i < in.nf; ++i) bulk = bulk && aligned(in.fin[i], 16);
      for (int i = 0; i < in.nb; ++i) bulk = bulk && aligned(in.bin[i], 16);
    }
  }
  Plan p;
  if (!make_plan(kind, E, (int)T, A, flags, sm, vec_ok && T % 4 == 0, &p, bulk)) return RLCA_ERR_INVALID_ARG;
  if (p.ws_bytes > 0 && (ws == nullptr || ws_bytes < p.ws_bytes || !aligned(ws, 16))) return RLCA_ERR_INVALID_ARG;
  Geom g;
  g.E = E;
  g.T = (int)T;
  g.seg_len = p.seg_len;
  g.nseg = p.nseg;
  g.mode = kModeFull;
  g.vec = (!p.time_major && vec_ok && T % 4 == 0) ? 1 : 0;
  g.early = (flags & RLCA_INPUTS_READY) ? 1 : 0;
  g.ws = ws;
  g.aux = p.aux_bytes > 0 ? reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + aux_offset(p.ws_bytes, p.aux_bytes))
                          : nullptr;
  if (run_scan(est, p, g, s) != cudaSuccess) return RLCA_ERR_CUDA;
  return checked_build_status(s);
}

}  // namespace

bool make_plan(Kind kind, int64_t E, int T, int num_actions, uint32_t flags, int sm_count, bool vec,
               Plan* out, bool bulk) {
  const bool retrace = kind == Kind::Retrace;
  Plan q = {};
  q.time_major = (flags & RLCA_TIME_MAJOR) != 0;
  const bool bf16_io = (flags & RLCA_BF16) != 0;
  if (q.time_major) {
    // Retrace: 8 chunk warps keep two CTAs' staging buffers on an SM; 16
    // where the environments give at most one CTA per SM anyway -- unless
    // rows of more than one 128-step tile would, at 8, split into two-pass
    // segments (more CTAs), a split the wider CTAs would no longer take
    int cmax = kTmMaxWidth;
    if (retrace) {
      const int64_t rb = (E + 31) / 32;
      const bool c8_splits = T > 64 && 16 * rb * 256 < (int64_t)sm_count * 1024;
      cmax = rb <= sm_count && (!c8_splits || T <= 128) ? kRetraceTmMaxWidth : kRetraceTmMaxWidth / 2;
    }
    int C = (int)std::min<int64_t>(next_pow2((T + 7) / 8), cmax);
    if (flags & RLCA_MULTIPASS) C = std::max(1, C / 4);
    // Retrace's per-warp staging grows with A: fewer chunk warps when it would not fit
    while (retrace && C > 1 &&
           (size_t)C * retrace_raw_floats(num_actions, true) * 4 + (size_t)3 * (8 * C + 1) * 32 * 4 +
                   (size_t)2 * C * 32 * kMaxMapBytes > kMaxSmemPerCta)
      C /= 2;
    q.width = C;
    q.block = 32 * C;
    q.rows_per_cta = 32;
    q.tile = 8 * C;
    q.smem_driver_bound = (size_t)2 * C * 32 * kMaxMapBytes;
    q.smem = retrace ? (size_t)C * retrace_raw_floats(num_actions, true) * 4 + (size_t)3 * (q.tile + 1) * 32 * 4 : 0;
  } else {
    const int wmax = retrace ? kRetraceEmMaxWidth : kEmMaxWidth;
    int W = (int)std::min<int64_t>(next_pow2(std::max<int64_t>((T + kEmSteps - 1) / kEmSteps, kEmMinWidth)),
                                   wmax);
    if (flags & RLCA_MULTIPASS) W = std::max(kEmMinWidth, W / 4);
    q.width = W;
    q.block = std::max(W, kEmMinBlock);
    q.rows_per_cta = q.block / W;
    q.tile = kEmSteps * W;
    const int nwr = W > 32 ? W / 32 : 1;
    q.smem_driver_bound = nwr > 1 ? (size_t)2 * q.rows_per_cta * nwr * kMaxMapBytes : 0;
    q.smem = retrace ? (size_t)(q.block / 32) * retrace_raw_floats(num_actions, false) * 4 +
                         (size_t)3 * q.rows_per_cta * (q.tile + 1) * 4
                     : 0;
  }
  q.ntiles = (int)((T + q.tile - 1) / q.tile);
  q.row_blocks = (E + q.rows_per_cta - 1) / q.rows_per_cta;
  int nseg = 1;
  if (flags & RLCA_MULTIPASS) {
    nseg = q.ntiles >= 2 ? (q.ntiles + 1) / 2 : 1;
  } else {
    // split long rows across CTAs only when the rows alone leave the GPU
    // mostly idle; the second pass re-reads the inputs (for Retrace, 161
    // bytes a step: it splits only when the rows are 8x fewer still)
    const int64_t threads = q.row_blocks * q.block;
    const int64_t target = (int64_t)sm_count * 1024;
    if (q.ntiles > 1 && 2 * threads < target && (!retrace || 16 * threads < target)) {
      nseg = (int)std::min<int64_t>(q.ntiles, (target + threads - 1) / threads);
      // Retrace CTAs are held to a few an SM by their staging buffers:
      // split to that many CTAs rather than to a thread count
      if (retrace && kRetraceSplitCtasPerSm > 0)
        nseg = (int)std::min<int64_t>(
            q.ntiles, ((int64_t)kRetraceSplitCtasPerSm * sm_count + q.row_blocks - 1) / q.row_blocks);
    }
  }
  const int seg_tiles = (q.ntiles + nseg - 1) / nseg;
  q.seg_len = seg_tiles * q.tile;
  q.nseg = (q.ntiles + seg_tiles - 1) / seg_tiles;
  // one affine map per (row, segment): two values, two of each for the fused value targets
  const size_t ws_elem = kind == Kind::ValueTargets ? 16 : 8;
  q.ws_bytes = q.nseg > 1 ? (size_t)E * q.nseg * ws_elem : 0;
  // Retrace's two passes: the first also leaves every step's (E_pi Q, Q(a),
  // c) in three float planes after the maps (256-byte aligned), so the
  // second reads 12 bytes a step instead of the 2 A values of Q and pi
  q.aux_bytes = 0;
  if (retrace && q.nseg > 1) {
    q.ws_bytes = (q.ws_bytes + 255) & ~size_t(255);
    q.aux_bytes = (size_t)3 * (size_t)E * (size_t)T * sizeof(float);
    q.ws_bytes += q.aux_bytes;
  }
  const bool fast_ok = !q.time_major && vec && q.nseg == 1 && !(flags & RLCA_MULTIPASS);
  q.fast = fast_ok && T % kEmSteps == 0 && q.ntiles == 1;
  q.steps = kEmSteps;
  // 8 steps a thread (half the warps and scan rounds a row) where the
  // threads still fill the GPU: rows of >= 1024 steps (Retrace, whose
  // per-warp staging keeps fewer CTAs resident, at four times the threads);
  // float32 rows of 256-1023 steps at twice the threads; bfloat16 rows from
  // 64 steps on (one 16-byte vector per array, the bytes a float32 thread
  // moves with 4).  V-Trace, whose four inputs cost occupancy, takes only
  // the first rule.
  const int W8 = next_pow2((T + 7) / 8);
  const int64_t l8_min_threads = (int64_t)sm_count * 1024 * (retrace ? 4 : 1);
  const int l8_min_t = (bf16_io && kind != Kind::Vtrace) ? 64 : kFastL8MinT;
  // (float32 V-Trace stays at 4 steps: at 8 it holds 67-80 registers, and
  // 4 measured faster at T = 2048, 0.78 against 0.75 of the bandwidth)
  const bool l8 = ((kind != Kind::Vtrace || bf16_io) && T >= l8_min_t && (int64_t)E * (T / 8) >= l8_min_threads) ||
                  (!bf16_io && kind != Kind::Vtrace && T >= 256 && (int64_t)E * (T / 8) >= 2 * l8_min_threads);
  if (fast_ok && l8 && T % 8 == 0 && W8 <= (retrace ? kRetraceEmMaxWidth : kEmMaxWidth)) {
    q.fast = true;
    q.steps = 8;
    q.ntiles = 1;
    q.width = W8;
    q.block = std::max(W8, kEmMinBlock);
    q.rows_per_cta = q.block / W8;
    q.tile = 8 * W8;
    q.row_blocks = (E + q.rows_per_cta - 1) / q.rows_per_cta;
    q.seg_len = q.tile;
    q.smem_driver_bound = W8 > 32 ? (size_t)2 * q.rows_per_cta * (W8 / 32) * kMaxMapBytes : 0;
    if (retrace)
      q.smem = (size_t)(q.block / 32) * retrace_raw_floats(num_actions, false) * 4 +
               (size_t)3 * q.rows_per_cta * (q.tile + 1) * 4;
  }
  // time-major rows of whole 8-step chunks with 32-bit element offsets take
  // the fast time-major drivers: 32 environments per CTA once that still
  // leaves two CTAs per SM, else one 32-byte sector of a step row (8 float32
  // or 16 bfloat16 environments; more CTAs); few environments with long rows
  // split them into segments (two passes).
  const int ct_need = next_pow2((T + 7) / 8);
  // narrow CTAs read one 32-byte sector of a step row: 8 float32 or 16 bfloat16 environments
  const int tf_ew = (E >= (int64_t)64 * sm_count || ct_need < 4) ? 32 : (bf16_io ? 16 : 8);
  const int tf_ct = std::min(ct_need, tf_ew == 32 ? 16 : 32);
  if (q.time_major && !retrace && T % 8 == 0 && !(flags & RLCA_MULTIPASS) &&
      (uint64_t)E * (uint64_t)T < (uint64_t{1} << 32)) {
    // staged: the step rows stream through a shared-memory ring in 16-byte
    // pieces (E a multiple of the environments per piece, aligned inputs):
    // rows of 32 environments in 64-step tiles; for the one-float-input
    // scans also rows of 16.  Otherwise the rows go straight into registers.
    const bool staged32 = kTmStaged && vec && E % (bf16_io ? 8 : 4) == 0 && tf_ew == 32;
    // (with two or more float inputs the direct 8-environment driver measured faster)
    const bool one_float = kind == Kind::Disc || kind == Kind::Elig || kind == Kind::PrefixSum;
    const bool staged16 = kTmStaged16 && one_float && vec && !bf16_io && E % 4 == 0 && tf_ew == 8;
    bool staged = staged32 || staged16;
    int EW = staged16 ? 16 : tf_ew;
    int CT = staged32 ? std::min(tf_ct, 8) : tf_ct;
    // bulk: each tile of each input is one tensor copy into a ring of
    // RLCA_TB_STAGES stages, 32 environments per CTA once E gives two such
    // CTAs per SM, else 8 (below); chunk-threads so the ring stays within
    // kTbRingBytes and a CTA within 256 threads.  (16-environment CTAs,
    // split into two passes or not, measured slower than the direct
    // 8-environment driver.)
    const StageCounts sc = stage_counts(kind);
    const bool wide = E >= (int64_t)kTbMinEnvsPerSm * sm_count;
    // 8-environment tiles (one 32-byte sector of a float32 step row, the
    // flag rows copied 16 environments wide) where they pay: two or more
    // float inputs, rows of several 256-step tiles, and enough CTAs of 8
    // environments that rows stay whole (one pass).  Measured against the
    // direct driver at 4096 x 2048: 1.08-1.13x; at 4096 x 128-512, with
    // one float input, or split into two passes: 0.65-1.0x.
    const int narrow_ct = std::max(4, std::min(ct_need, 32));
    const bool narrow = kTbNarrow && !bf16_io && sc.nf >= 2 && (E / 8) >= (int64_t)kTbCtasPerSm * sm_count &&
                        (T + 8 * narrow_ct - 1) / (8 * narrow_ct) >= kTbNarrowMinTiles;
    if (kTmBulk && bulk && E % 16 == 0 && (wide || narrow)) {
      EW = wide ? 32 : 8;
      const size_t row_bytes = (size_t)sc.nf * (bf16_io ? 2 : 4) * EW + (size_t)sc.nb * (EW < 16 ? 16 : EW);
      const int ct_min = 32 / EW;  // whole warps
      CT = std::max(ct_min, std::min(ct_need, 256 / EW));
      while (CT > ct_min && (size_t)RLCA_TB_STAGES * 8 * CT * row_bytes > kTbRingBytes) CT /= 2;
      staged = false;
      q.tm_bulk = true;
    }
    q.tm_fast = true;
    q.tm_staged = staged;
    q.env_width = EW;
    q.width = CT;
    q.block = EW * CT;
    q.rows_per_cta = EW;
    q.tile = 8 * CT;
    q.ntiles = (T + q.tile - 1) / q.tile;
    q.row_blocks = (E + EW - 1) / EW;
    // the two-pass split when the environments alone leave the GPU mostly
    // idle and each would walk more than four tiles (a shorter walk costs
    // less than the second read of the inputs)
    const int64_t threads = q.row_blocks * q.block;
    const int64_t target = (int64_t)sm_count * 1024;
    int ns = 1;
    if (q.tm_bulk) {
      // the bulk driver keeps its tiles in flight by copies, not threads:
      // split rows across CTAs until there are kTbCtasPerSm CTAs an SM (a
      // second pass re-reads the inputs, from L2 while they fit there)
      const int64_t want = (int64_t)kTbCtasPerSm * sm_count;
      if (q.ntiles > 1 && q.row_blocks < want)
        ns = (int)std::min<int64_t>(q.ntiles, (want + q.row_blocks - 1) / q.row_blocks);
    } else if (q.ntiles > 4 && 2 * threads < target) {
      ns = (int)std::min<int64_t>(q.ntiles, (target + threads - 1) / threads);
    }
    const int seg_tiles = (q.ntiles + ns - 1) / ns;
    q.seg_len = seg_tiles * q.tile;
    q.nseg = (q.ntiles + seg_tiles - 1) / seg_tiles;
    q.ws_bytes = q.nseg > 1 ? (size_t)E * q.nseg * ws_elem : 0;
    q.smem = 0;
    q.smem_driver_bound = (size_t)CT * (EW + 1) * (kMaxMapBytes + kMaxMapBytes / 2);
    // the stages: at most 4 float and 2 flag inputs of CT * (8 * EW + EW) elements
    if (staged) q.smem_driver_bound += (size_t)RLCA_TS_STAGES * ((size_t)CT * 9 * EW * 18 + 16);
    // barriers, alignment slack and the tensor-copy ring
    if (q.tm_bulk)
      q.smem_driver_bound +=
          256 + (size_t)RLCA_TB_STAGES * 8 * CT * ((size_t)sc.nf * (bf16_io ? 2 : 4) * EW + (size_t)sc.nb * (EW < 16 ? 16 : EW));
  }
  if (q.row_blocks * q.nseg > INT32_MAX) return false;
  if (q.smem + q.smem_driver_bound > kMaxSmemPerCta) return false;

  *out = q;
  return true;
}

bool retrace_tail_plan(const Plan& p, int64_t E, int T, bool two_byte, Plan* out) {
  if (!p.time_major || p.nseg < 2 || T % 8 != 0 || (uint64_t)E * (uint64_t)T >= (uint64_t{1} << 32)) return false;
  const int EW = two_byte ? 16 : 8;  // one 32-byte sector of a step row
  int CT = 32;
  while (CT > 1 && p.seg_len % (8 * CT) != 0) CT /= 2;
  if (EW * CT < 32 || p.seg_len % (8 * CT) != 0) return false;  // whole warps
  Plan q = p;
  q.fast = false;
  q.tm_fast = true;
  q.tm_staged = false;
  q.tm_bulk = false;
  q.env_width = EW;
  q.width = CT;
  q.block = EW * CT;
  q.rows_per_cta = EW;
  q.tile = 8 * CT;
  q.ntiles = (T + q.tile - 1) / q.tile;
  q.row_blocks = (E + EW - 1) / EW;
  q.smem = 0;
  q.smem_driver_bound = (size_t)CT * (EW + 1) * (kMaxMapBytes + kMaxMapBytes / 2);
  if (q.row_blocks * q.nseg > INT32_MAX) return false;
  *out = q;
  return true;
}

StageCounts stage_counts(Kind kind) {
  switch (kind) {
    case Kind::Gae:
    case Kind::TdLambda:
    case Kind::ValueTargets: return {2, 2};
    case Kind::Disc:
    case Kind::Elig:
    case Kind::PrefixSum: return {1, 2};
    case Kind::Vtrace: return {4, 2};
    case Kind::Affine: return {2, 0};
    default: return {0, 0};
  }
}

namespace {

// the driver's tensor-map encoder, reached through the runtime's entry-point
// query (the library links only the runtime)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// [T, E] array of elem_bytes elements, E innermost; boxes of ew x rows; the
// copy moves bits, so the element type only gives the size
bool encode_2d(CUtensorMap* m, const void* base, int elem_bytes, int64_t E, int64_t T, int ew, int rows) {
  const EncodeTiledFn fn = encoder();
  if (fn == nullptr) return false;
  const CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT32;
  const cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)T};
  const cuuint64_t strides[1] = {(cuuint64_t)E * (cuuint64_t)elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)ew, (cuuint32_t)rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tensor_maps_available() { return encoder() != nullptr; }

bool encode_tm_maps(const StagedList& in, int elem_bytes, int64_t E, int64_t T, int ew, int rows, TmaSet* out) {
  for (int i = 0; i < in.nf; ++i)
    if (!encode_2d(&out->f[i], in.fin[i], elem_bytes, E, T, ew, rows)) return false;
  for (int i = 0; i < in.nb; ++i)
    if (in.bin[i] != nullptr && !encode_2d(&out->b[i], in.bin[i], 1, E, T, ew < 16 ? 16 : ew, rows)) return false;
  return true;
}

}  // namespace rlca

using namespace rlca;

extern "C" {

const char* rlca_status_string(int status) {
  switch (status) {
    case RLCA_OK: return "ok";
    case RLCA_ERR_INVALID_ARG: return "invalid argument";
    case RLCA_ERR_UNSUPPORTED: return "unsupported argument";
    case RLCA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int rlca_version(void) { return 200; }

int rlca_index_checks(void) { return kIndexCheck ? 1 : 0; }

int rlca_device_status(unsigned int* status, int clear) {
  if (status == nullptr) return RLCA_ERR_INVALID_ARG;
  *status = 0;
  const bool c = clear != 0;
  cudaError_t (*const units[])(unsigned int*, bool) = {status_values, status_values_bf16_a, status_values_bf16_b,
                                                       status_offpolicy, status_offpolicy_bf16, status_forward,
                                                       status_forward_bf16};
  for (auto f : units)
    if (f(status, c) != cudaSuccess) return RLCA_ERR_CUDA;
  return RLCA_OK;
}

int rlca_workspace_size(int estimator, int64_t E, int64_t T, int32_t num_actions, uint32_t flags, size_t* bytes) {
  if (bytes == nullptr) return RLCA_ERR_INVALID_ARG;
  *bytes = 0;
  Kind kind;
  switch (estimator) {
    case RLCA_EST_GAE: kind = Kind::Gae; break;
    case RLCA_EST_DISCOUNTED_RETURN: kind = Kind::Disc; break;
    case RLCA_EST_TD_LAMBDA: kind = Kind::TdLambda; break;
    case RLCA_EST_VTRACE: kind = Kind::Vtrace; break;
    case RLCA_EST_RETRACE: kind = Kind::Retrace; break;
    case RLCA_EST_ELIG_TRACE: kind = Kind::Elig; break;
    case RLCA_EST_PREFIX_SUM: kind = Kind::PrefixSum; break;
    case RLCA_EST_AFFINE_SCAN: kind = Kind::Affine; break;
    case RLCA_EST_VALUE_TARGETS: kind = Kind::ValueTargets; break;
    default: return RLCA_ERR_INVALID_ARG;
  }
  const uint32_t allowed =
      kFloatFlags | (kind == Kind::PrefixSum ? (RLCA_PSUM_EXCLUSIVE | RLCA_PSUM_FLAG_IS_START) : 0u);
  if (!flags_ok(flags, allowed)) return RLCA_ERR_INVALID_ARG;
  if (kind == Kind::Retrace && num_actions < 1) return RLCA_ERR_INVALID_ARG;
  if (kind == Kind::Retrace && num_actions > RLCA_MAX_ACTIONS) return RLCA_ERR_UNSUPPORTED;
  int st;
  if (check_sizes(E, T, &st)) return st;
  int sm = 0;
  if (sm_count_of_current_device(&sm) != cudaSuccess) return RLCA_ERR_CUDA;
  // the call picks the staged or the direct path from its pointers' alignment,
  // which the query cannot see: report the larger of the two needs
  Plan pd, ps, pb;
  if (!make_plan(kind, E, (int)T, num_actions, flags & kFloatFlags, sm, false, &pd)) return RLCA_ERR_INVALID_ARG;
  if (!make_plan(kind, E, (int)T, num_actions, flags & kFloatFlags, sm, true, &ps)) return RLCA_ERR_INVALID_ARG;
  if (!make_plan(kind, E, (int)T, num_actions, flags & kFloatFlags, sm, true, &pb, true)) return RLCA_ERR_INVALID_ARG;
  *bytes = std::max(std::max(pd.ws_bytes, ps.ws_bytes), pb.ws_bytes);
  return RLCA_OK;
}

int rlca_gae(const float* rewards, const float* values, const uint8_t* terminated, const uint8_t* truncated,
             const float* trunc_value, const float* bootstrap, float* advantages, float* returns, int64_t E,
             int64_t T, float gamma, float lambda, uint32_t flags, void* workspace, size_t workspace_bytes,
             rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !values || !advantages || (truncated && !trunc_value)) return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T);
  if (any_overlap({{rewards, nf}, {values, nf}, {terminated, nb}, {truncated, nb}, {trunc_value, nf},
                   {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{advantages, nf}, {returns, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(values, 16) && aligned(advantages, 16) &&
                   aligned(returns, 16) && aligned(terminated, 4) && aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    auto fill = [&](auto& e) {
      e.b = b; e.r = rewards; e.v = values; e.adv = advantages; e.ret = returns; e.gamma = gamma;
      e.gl = gamma * lambda;
    };
    if (truncated) {
      GaeEst<true, ST> e;
      fill(e);
      return launch(Kind::Gae, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    GaeEst<false, ST> e;
    fill(e);
    return launch(Kind::Gae, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_value_targets(const float* rewards, const float* values, const uint8_t* terminated,
                       const uint8_t* truncated, const float* trunc_value, const float* bootstrap, float* advantages,
                       float* returns, float* disc_returns, float* td_lambda_returns, int64_t E, int64_t T,
                       float gamma, float lambda, uint32_t flags, void* workspace, size_t workspace_bytes,
                       rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !values || (truncated && !trunc_value)) return RLCA_ERR_INVALID_ARG;
  if (!advantages && !returns && !disc_returns && !td_lambda_returns) return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T);
  if (any_overlap({{rewards, nf}, {values, nf}, {terminated, nb}, {truncated, nb}, {trunc_value, nf},
                   {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{advantages, nf}, {returns, nf}, {disc_returns, nf}, {td_lambda_returns, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(values, 16) && aligned(advantages, 16) &&
                   aligned(returns, 16) && aligned(disc_returns, 16) && aligned(td_lambda_returns, 16) &&
                   aligned(terminated, 4) && aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    auto fill = [&](auto& e) {
      e.b = b; e.r = rewards; e.v = values; e.adv = advantages; e.ret = returns; e.disc = disc_returns;
      e.td = td_lambda_returns; e.gamma = gamma; e.gl = gamma * lambda;
    };
    if (truncated) {
      ValueTargetsEst<true, ST> e;
      fill(e);
      return launch(Kind::ValueTargets, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    ValueTargetsEst<false, ST> e;
    fill(e);
    return launch(Kind::ValueTargets, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_discounted_return(const float* rewards, const uint8_t* terminated, const uint8_t* truncated,
                           const float* trunc_value, const float* bootstrap, float* returns, int64_t E, int64_t T,
                           float gamma, uint32_t flags, void* workspace, size_t workspace_bytes,
                           rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !returns || (truncated && !trunc_value)) return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T);
  if (any_overlap({{rewards, nf}, {terminated, nb}, {truncated, nb}, {trunc_value, nf},
                   {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{returns, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(returns, 16) && aligned(terminated, 4) && aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    if (truncated) {
      DiscEst<true, ST> e;
      e.b = b; e.r = rewards; e.out = returns; e.gamma = gamma;
      return launch(Kind::Disc, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    DiscEst<false, ST> e;
    e.b = b; e.r = rewards; e.out = returns; e.gamma = gamma;
    return launch(Kind::Disc, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_td_lambda(const float* rewards, const float* values, const uint8_t* terminated, const uint8_t* truncated,
                   const float* trunc_value, const float* bootstrap, float* returns, int64_t E, int64_t T,
                   float gamma, float lambda, uint32_t flags, void* workspace, size_t workspace_bytes,
                   rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !values || !returns || (truncated && !trunc_value)) return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T);
  if (any_overlap({{rewards, nf}, {values, nf}, {terminated, nb}, {truncated, nb}, {trunc_value, nf},
                   {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{returns, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(values, 16) && aligned(returns, 16) && aligned(terminated, 4) &&
                   aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    auto fill = [&](auto& e) {
      e.b = b; e.r = rewards; e.v = values; e.out = returns; e.gamma = gamma; e.gl = gamma * lambda;
      e.one_minus_lambda = 1.f - lambda;
    };
    if (truncated) {
      TdLambdaEst<true, ST> e;
      fill(e);
      return launch(Kind::TdLambda, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    TdLambdaEst<false, ST> e;
    fill(e);
    return launch(Kind::TdLambda, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_vtrace(const float* rewards, const float* values, const float* logp_target, const float* logp_behaviour,
                const uint8_t* terminated, const uint8_t* truncated, const float* trunc_value,
                const float* bootstrap, float* vs, float* pg_advantages, int64_t E, int64_t T, float gamma,
                float rho_bar, float c_bar, float lambda, uint32_t flags, void* workspace, size_t workspace_bytes,
                rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!rewards || !values || !logp_target || !logp_behaviour || !vs || (truncated && !trunc_value))
    return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T);
  if (any_overlap({{rewards, nf}, {values, nf}, {logp_target, nf}, {logp_behaviour, nf}, {terminated, nb},
                   {truncated, nb}, {trunc_value, nf}, {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{vs, nf}, {pg_advantages, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(values, 16) && aligned(logp_target, 16) &&
                   aligned(logp_behaviour, 16) && aligned(vs, 16) && aligned(pg_advantages, 16) &&
                   aligned(terminated, 4) && aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    auto fill = [&](auto& e) {
      e.b = b; e.r = rewards; e.v = values; e.lpt = logp_target; e.lpb = logp_behaviour; e.vs = vs;
      e.pg = pg_advantages; e.gamma = gamma; e.rho_bar = rho_bar; e.c_bar = c_bar; e.lambda = lambda;
    };
    if (truncated) {
      VtraceEst<true, ST> e;
      fill(e);
      return launch(Kind::Vtrace, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    VtraceEst<false, ST> e;
    fill(e);
    return launch(Kind::Vtrace, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_retrace(const float* q, const float* pi, const float* mu_a, const int32_t* actions, const float* rewards,
                 const uint8_t* terminated, const uint8_t* truncated, const float* trunc_value,
                 const float* bootstrap, float* q_ret, int64_t E, int64_t T, int32_t num_actions, float gamma,
                 float lambda, uint32_t flags, void* workspace, size_t workspace_bytes, rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (num_actions < 1) return RLCA_ERR_INVALID_ARG;
  if (num_actions > RLCA_MAX_ACTIONS) return RLCA_ERR_UNSUPPORTED;
  if (!q || !pi || !mu_a || !actions || !rewards || !q_ret || (truncated && !trunc_value))
    return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe, nb = (size_t)(E * T), nq = nf * (size_t)num_actions;
  if (any_overlap({{q, nq}, {pi, nq}, {mu_a, nf}, {actions, (size_t)(E * T) * 4}, {rewards, nf}, {terminated, nb},
                   {truncated, nb}, {trunc_value, nf}, {bootstrap, (size_t)E * fe}, {workspace, workspace_bytes}},
                  {{q_ret, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(rewards, 16) && aligned(q_ret, 16) && aligned(terminated, 4) && aligned(truncated, 4);
  const BoundaryArgs b{terminated, truncated, trunc_value, bootstrap, (int)T};
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    const RetraceStage<ST> stg{q, pi, mu_a, actions, num_actions, lambda, E * T};
    if (truncated) {
      RetraceEst<true, ST> e;
      e.b = b; e.st = stg; e.r = rewards; e.out = q_ret; e.gamma = gamma;
      return launch(Kind::Retrace, e, E, T, num_actions, flags, workspace, workspace_bytes, vec, stream);
    }
    RetraceEst<false, ST> e;
    e.b = b; e.st = stg; e.r = rewards; e.out = q_ret; e.gamma = gamma;
    return launch(Kind::Retrace, e, E, T, num_actions, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_elig_trace(const float* x, const uint8_t* terminated, const uint8_t* truncated, float* out, int64_t E,
                    int64_t T, float gamma, float lambda, uint32_t flags, void* workspace, size_t workspace_bytes,
                    rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!x || !out) return RLCA_ERR_INVALID_ARG;
  const size_t nf = (size_t)(E * T) * fbytes(flags), nb = (size_t)(E * T);
  if (any_overlap({{x, nf}, {terminated, nb}, {truncated, nb}, {workspace, workspace_bytes}}, {{out, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(x, 16) && aligned(out, 16) && aligned(terminated, 4) && aligned(truncated, 4);
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    EligEst<ST> e;
    e.x = x; e.term = terminated; e.trunc = truncated; e.out = out; e.gl = gamma * lambda;
    return launch(Kind::Elig, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_episodic_prefix_sum(const void* x, int dtype, const uint8_t* terminated, const uint8_t* truncated,
                             void* out, int64_t E, int64_t T, uint32_t flags, void* workspace,
                             size_t workspace_bytes, rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags | RLCA_PSUM_EXCLUSIVE | RLCA_PSUM_FLAG_IS_START)) return RLCA_ERR_INVALID_ARG;
  if (dtype != RLCA_F32 && dtype != RLCA_I32) return RLCA_ERR_INVALID_ARG;
  if (dtype == RLCA_I32 && (flags & RLCA_BF16)) return RLCA_ERR_INVALID_ARG;
  if (!x || !out) return RLCA_ERR_INVALID_ARG;
  const size_t nf = (size_t)(E * T) * fbytes(flags), nb = (size_t)(E * T);
  if (any_overlap({{x, nf}, {terminated, nb}, {truncated, nb}, {workspace, workspace_bytes}}, {{out, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(x, 16) && aligned(out, 16) && aligned(terminated, 4) && aligned(truncated, 4);
  const uint32_t core = flags & kFloatFlags;
  const int excl = (flags & RLCA_PSUM_EXCLUSIVE) ? 1 : 0;
  const int start = (flags & RLCA_PSUM_FLAG_IS_START) ? 1 : 0;
  if (dtype == RLCA_I32) {
    PrefixSumEst<uint32_t> e;
    e.x = x; e.term = terminated; e.trunc = truncated; e.out = out; e.exclusive = excl; e.flag_is_start = start;
    return launch(Kind::PrefixSum, e, E, T, 0, core, workspace, workspace_bytes, vec, stream);
  }
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    PrefixSumEst<float, ST> e;
    e.x = x; e.term = terminated; e.trunc = truncated; e.out = out; e.exclusive = excl; e.flag_is_start = start;
    return launch(Kind::PrefixSum, e, E, T, 0, core, workspace, workspace_bytes, vec, stream);
  });
}

int rlca_affine_scan(const float* alpha, const float* beta, const float* carry, float* out, int64_t E, int64_t T,
                     int reverse, uint32_t flags, void* workspace, size_t workspace_bytes, rlca_stream_t stream) {
  int st;
  if (check_sizes(E, T, &st)) return st;
  if (!flags_ok(flags, kFloatFlags)) return RLCA_ERR_INVALID_ARG;
  if (!alpha || !beta || !out) return RLCA_ERR_INVALID_ARG;
  const size_t fe = fbytes(flags), nf = (size_t)(E * T) * fe;
  if (any_overlap({{alpha, nf}, {beta, nf}, {carry, (size_t)E * fe}, {workspace, workspace_bytes}}, {{out, nf}}))
    return RLCA_ERR_INVALID_ARG;
  const bool vec = aligned(alpha, 16) && aligned(beta, 16) && aligned(out, 16);
  return with_storage(flags, [&](auto tag) {
    using ST = typename decltype(tag)::type;
    if (reverse) {
      AffineEst<true, ST> e;
      e.alpha = alpha; e.beta = beta; e.carry = carry; e.out = out;
      return launch(Kind::Affine, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
    }
    AffineEst<false, ST> e;
    e.alpha = alpha; e.beta = beta; e.carry = carry; e.out = out;
    return launch(Kind::Affine, e, E, T, 0, flags, workspace, workspace_bytes, vec, stream);
  });
}

}  // extern "C"
