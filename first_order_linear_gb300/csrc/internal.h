// internal.h -- host-side launch planning shared by the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "drivers.cuh"

namespace rlca {

enum class Kind { Gae, Disc, TdLambda, Vtrace, Retrace, Elig, PrefixSum, Affine, ValueTargets };

// Largest env-major threads-per-row and time-major chunk-threads per
// environment of a kind (Retrace keeps its tiles small: it stages its
// per-action blocks in shared memory).
constexpr int kEmMaxWidth = 1024;
constexpr int kTmMaxWidth = 32;
constexpr int kRetraceEmMaxWidth = 256;
constexpr int kRetraceTmMaxWidth = 16;
constexpr int kEmMinWidth = 1;
constexpr size_t kMaxSmemPerCta = 227 * 1024;

struct Plan {
  bool time_major;
  bool fast;        // env-major, one tile per row, one segment (em_fast_kernel)
  bool tm_fast;     // time-major, T % 8 == 0, E * T < 2^32, one segment (tm_fast_kernel)
  bool tm_staged;   // ... and inputs staged through shared memory (tm_staged_kernel)
  bool tm_bulk;     // ... staged by tensor-memory-accelerator tile copies (tm_bulk_kernel)
  int steps;        // steps per thread of the fast driver (kEmSteps or 8)
  int width;        // env-major: threads per row; time-major: chunk-threads per environment
  int env_width;    // fast time-major: environments per CTA (8 or 32)
  int block;        // threads per CTA
  int rows_per_cta;
  int tile;         // steps per tile
  int ntiles;       // tiles per row
  int nseg;         // segments per row (> 1: two-pass)
  int seg_len;      // steps per segment
  int64_t row_blocks;
  size_t smem;      // estimator staging shared memory per CTA (the launcher adds the driver's exchange arrays)
  size_t smem_driver_bound;  // upper bound of the driver's part, for the size check
  size_t ws_bytes;  // workspace of the two-pass path (segment maps, then aux_bytes)
  size_t aux_bytes; // Retrace's per-step scalar planes at the workspace's end (two-pass path)
};

// byte offset of the Retrace scalar planes inside a two-pass workspace
constexpr size_t aux_offset(size_t ws_bytes, size_t aux_bytes) { return ws_bytes - aux_bytes; }

// Fills *p for a problem; returns false when the sizes cannot be launched.
// vec: the env-major arrays are 16-byte aligned (4-byte for flags) and
// T % 4 == 0, so rows can be read as 16-byte vectors.  bulk: every staged
// input starts on a 16-byte boundary, E % 16 == 0 and the tensor-map encoder
// is available, so time-major tiles may move by tensor copies.
bool make_plan(Kind kind, int64_t E, int T, int num_actions, uint32_t flags, int sm_count, bool vec, Plan* p,
               bool bulk = false);

// The second pass of Retrace's time-major two-pass split on the fast
// time-major driver (RetraceTailEst): the first pass's segments (nseg,
// seg_len) in CTAs of 8 environments (16 for 2-byte storage) and CT chunk
// threads, CT the largest power of two up to 32 whose 8 * CT steps divide a
// segment.  False where that driver does not apply (env-major, one
// segment, T % 8 != 0, E * T >= 2^32); the first pass's kernel then runs
// the second as well.
bool retrace_tail_plan(const Plan& p, int64_t E, int T, bool two_byte, Plan* out);

// bytes a time-major step stages per staged input set (float inputs of
// fbytes each, flag inputs of one byte)
struct StageCounts {
  int nf, nb;
};
StageCounts stage_counts(Kind kind);

// The 2-D tensor maps of a call's staged time-major inputs ([T, E], E
// innermost; tiles of ew environments x rows steps, flag tiles at least 16
// environments wide).  False when the encoder is unavailable or refuses a
// map.
bool encode_tm_maps(const StagedList& in, int elem_bytes, int64_t E, int64_t T, int ew, int rows, TmaSet* out);
// whether encode_tm_maps can work at all (the driver's encoder was found)
bool tensor_maps_available();

// RLCA_OK, or in the index-check build RLCA_ERR_CUDA once the stream's work
// has recorded a condition in a status word (it synchronises the stream)
int checked_build_status(cudaStream_t s);

// Reads (and with clear, zeroes) the device status word of each kernel
// translation unit, ORed into *word.  Synchronous copies.
cudaError_t status_values(unsigned int* word, bool clear);
cudaError_t status_values_bf16_a(unsigned int* word, bool clear);
cudaError_t status_values_bf16_b(unsigned int* word, bool clear);
cudaError_t status_offpolicy(unsigned int* word, bool clear);
cudaError_t status_offpolicy_bf16(unsigned int* word, bool clear);
cudaError_t status_forward(unsigned int* word, bool clear);
cudaError_t status_forward_bf16(unsigned int* word, bool clear);

#ifndef RLCA_TM_STAGED
#define RLCA_TM_STAGED 1
#endif
// build-time choice: aligned time-major inputs stream through shared memory
// (tm_staged_kernel) rather than straight into registers (tm_fast_kernel)
constexpr bool kTmStaged = RLCA_TM_STAGED != 0;
#ifndef RLCA_TM_STAGED16
#define RLCA_TM_STAGED16 1
#endif
// ... also for float32 tiles of 16 environments (rows of 64 bytes) where the
// direct driver would take 8
constexpr bool kTmStaged16 = RLCA_TM_STAGED16 != 0;
#ifndef RLCA_TM_BULK
#define RLCA_TM_BULK 1
#endif
// build-time choice: time-major tiles move by tensor copies (tm_bulk_kernel)
// where the inputs allow it
constexpr bool kTmBulk = RLCA_TM_BULK != 0;
#ifndef RLCA_TB_RING_BYTES
#define RLCA_TB_RING_BYTES (96 * 1024)
#endif
// shared memory the bulk driver's ring may take (two CTAs an SM)
constexpr size_t kTbRingBytes = RLCA_TB_RING_BYTES;
#ifndef RLCA_TB_CTAS_PER_SM
#define RLCA_TB_CTAS_PER_SM 2
#endif
// CTAs per SM below which the bulk driver splits rows into segments
constexpr int kTbCtasPerSm = RLCA_TB_CTAS_PER_SM;
#ifndef RLCA_TB_NARROW
#define RLCA_TB_NARROW 1
#endif
// build-time choice: below RLCA_TB_MIN_ENVS_PER_SM environments an SM,
// float32 time-major tiles of 8 environments move by tensor copies too
constexpr bool kTbNarrow = RLCA_TB_NARROW != 0;
// ... for rows of at least this many tiles
constexpr int kTbNarrowMinTiles = 4;
#ifndef RLCA_TB_MIN_ENVS_PER_SM
#define RLCA_TB_MIN_ENVS_PER_SM 64
#endif
// environments per SM from which time-major calls take the bulk driver
constexpr int kTbMinEnvsPerSm = RLCA_TB_MIN_ENVS_PER_SM;
#ifndef RLCA_RETRACE_SPLIT_CTAS_PER_SM
#define RLCA_RETRACE_SPLIT_CTAS_PER_SM 2
#endif
// Retrace's two-pass split: CTAs per SM to split rows into (0: by threads).
// Its staging buffers hold it to two CTAs an SM; splitting to that (rather
// than to a thread count) measured 0.55 against 0.50 of the bandwidth at
// 1024 x 2048 time-major, the same elsewhere
constexpr int kRetraceSplitCtasPerSm = RLCA_RETRACE_SPLIT_CTAS_PER_SM;

// Launches the scan of one estimator functor (both passes of the two-pass
// path when p.nseg > 1).  Defined by explicit instantiation in the family
// translation units.
template <class Est>
cudaError_t run_scan(const Est& est, const Plan& p, const Geom& g, cudaStream_t s);

}  // namespace rlca
