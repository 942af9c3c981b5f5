/*
 * rlca.h -- C ABI of the GB300 (sm_103a) credit-assignment scans.
 *
 * The operation behind every entry point is the first-order linear
 * recurrence of "rl-triton: High-Performance Triton GPU Kernels for
 * Reinforcement Learning Credit Assignment" (arXiv:2608.17641),
 * §1 Introduction and §3.1 Shared scan formulation:
 *
 *     backward:  A_t = alpha_t + beta_t * A_{t+1}      (A_T given)
 *     forward:   A_t = alpha_t + beta_t * A_{t-1}      (A_{-1} given)
 *
 * evaluated independently for each of E environment rows of T steps, with
 * each estimator's (alpha_t, beta_t) built on chip from raw rollout inputs
 * (§3.3 Algorithm-specific recurrences) and the episode-boundary rules of
 * §3.2 Episode-boundary semantics:
 *
 *   terminated[e,t] != 0  the episode ended at t: successor value 0, beta_t = 0.
 *   truncated[e,t]  != 0  the episode was cut at t: the successor value is the
 *                         caller's trunc_value[e,t], beta_t = 0.  Where both
 *                         flags are set, termination wins.
 *   t = T-1, no flag      the rollout window ends: the successor value is
 *                         bootstrap[e] (0 when bootstrap is NULL).
 *   forward scans         restart after a flagged step; no bootstrap.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers owned by the caller; the library keeps no
 *    reference after the call returns.  Inputs are read once, outputs are
 *    written once, every output element is written (steps after a boundary
 *    included).  Outputs must not overlap any input or each other.
 *  - Layout: env-major [E, T] (t fastest) by default; with RLCA_TIME_MAJOR
 *    every [E, T] array is [T, E] (e fastest) and every per-action array is
 *    [T, E, A] instead of [E, T, A].  Per-environment vectors (bootstrap,
 *    carry) are [E] in both layouts.  Arrays are dense and contiguous.
 *  - Element types: float32 values (bfloat16 with RLCA_BF16), uint8 flags
 *    (nonzero = set), int32 actions.  Any pointer alignment is accepted;
 *    16-byte aligned bases with T % 4 == 0 take the vectorised load paths
 *    (env-major rows; time-major rows staged through shared memory).
 *  - Sizes: 0 <= E <= 2^31-1, 0 <= T <= 2^30.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without synchronising.  No host or device memory is
 *    allocated by any entry point.  Kernels are launched with programmatic
 *    stream serialization: they may be scheduled while the previous kernel
 *    of the stream drains, but touch no memory before it has completed, so
 *    stream order is kept.
 *  - Workspace: an entry point may need device scratch for the two-pass
 *    segmented path (long rows on few environments, or RLCA_MULTIPASS).
 *    Query its size with rlca_workspace_size() using the same E, T,
 *    num_actions and flags, and pass a device buffer of at least that many
 *    bytes (16-byte aligned).  A NULL workspace is valid when the size is 0.
 *    The workspace is scratch: its contents on entry are ignored and on exit
 *    are unspecified; calls that share one workspace must not overlap on the
 *    GPU.
 *  - E == 0 or T == 0 returns RLCA_OK and enqueues nothing.
 *  - Errors: RLCA_ERR_INVALID_ARG (NULL required pointer, negative or
 *    oversized E/T, overlapping outputs, workspace too small or misaligned,
 *    unknown flags) and RLCA_ERR_UNSUPPORTED (num_actions above
 *    RLCA_MAX_ACTIONS, RLCA_BF16 where noted) are detected on the host
 *    before anything is enqueued.  RLCA_ERR_CUDA reports a failed CUDA runtime call (device
 *    query or launch); the CUDA error itself is left readable through
 *    cudaGetLastError()/cudaPeekAtLastError().
 *  - Entry points are thread-safe and hold no global state except a
 *    per-device cache of device attributes filled on first use.
 */
#ifndef RLCA_H
#define RLCA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *rlca_stream_t;

/* ---- status codes ------------------------------------------------------ */
#define RLCA_OK               0
#define RLCA_ERR_INVALID_ARG  1
#define RLCA_ERR_UNSUPPORTED  2
#define RLCA_ERR_CUDA         3

/* ---- flags (bitwise OR) -------------------------------------------------- */
/* Arrays are time-major [T, E] ([T, E, A]) instead of env-major [E, T]. */
#define RLCA_TIME_MAJOR          0x1u
/* Use the two-pass segmented path even where one pass would do (the library
 * picks it by itself for long rows on few environments).  Needs workspace. */
#define RLCA_MULTIPASS           0x2u
/* The caller asserts that this call's inputs were not written by the kernel
 * that precedes it on the stream (they were complete before that kernel was
 * enqueued).  The kernel may then read its inputs while the preceding kernel
 * is still running, and only waits for it before writing anything, so
 * back-to-back calls on independent batches overlap.  Without the flag a
 * call reads nothing before the preceding kernel has completed.  Ignored by
 * the two-pass path.  A false assertion gives wrong results (never an
 * out-of-bounds access). */
#define RLCA_INPUTS_READY        0x10u
/* Every floating-point array of the call -- per-step inputs and outputs and
 * the per-environment [E] vectors (bootstrap, carry) -- holds IEEE bfloat16
 * values (2 bytes each, the upper half of a float32) instead of float32; the
 * pointers keep their declared float type and point at the bfloat16 data.
 * Arithmetic and the scan state stay float32; each output is rounded to
 * nearest-even bfloat16 once.  Flags and int32 arrays are unchanged.  With
 * rlca_episodic_prefix_sum it applies to RLCA_F32 data only (RLCA_I32:
 * RLCA_ERR_INVALID_ARG); rlca_gae_static_scratch returns
 * RLCA_ERR_UNSUPPORTED.  With rlca_retrace it covers q, pi and mu_a as well
 * (the expectation and the ratio are formed in float32).  The paper defers bfloat16 I/O to future work and
 * keeps scans in float32 (rl-triton (arXiv:2608.17641) §9 Discussion and
 * Future Work; §4 Implementation, numerical requirements): only storage is
 * narrowed here. */
#define RLCA_BF16                0x20u
/* rlca_episodic_prefix_sum: output the sum over the steps BEFORE t in t's
 * episode instead of the inclusive sum. */
#define RLCA_PSUM_EXCLUSIVE      0x4u
/* rlca_episodic_prefix_sum: a flagged step is the FIRST step of a new
 * episode (default: a flagged step is the LAST step of its episode). */
#define RLCA_PSUM_FLAG_IS_START  0x8u

/* ---- estimator ids (for rlca_workspace_size) ---------------------------- */
#define RLCA_EST_GAE               1
#define RLCA_EST_DISCOUNTED_RETURN 2
#define RLCA_EST_TD_LAMBDA         3
#define RLCA_EST_VTRACE            4
#define RLCA_EST_RETRACE           5
#define RLCA_EST_ELIG_TRACE        6
#define RLCA_EST_PREFIX_SUM        7
#define RLCA_EST_AFFINE_SCAN       8
#define RLCA_EST_VALUE_TARGETS     9

/* ---- prefix-sum element types ------------------------------------------- */
#define RLCA_F32 0
#define RLCA_I32 1

/* Largest num_actions accepted by rlca_retrace. */
#define RLCA_MAX_ACTIONS 64

/* Human-readable text of a status code (static storage, never NULL). */
const char *rlca_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int rlca_version(void);

/* Device status bits (see rlca_device_status). */
#define RLCA_STATUS_WAIT_TIMEOUT 0x1u /* a bounded wait on a tile copy gave up */
#define RLCA_STATUS_INDEX        0x2u /* index-check build: an out-of-range index was skipped */

/*
 * Device-side status of the kernels launched so far on the CURRENT device:
 * writes to *status the OR of the status words the kernels keep in device
 * memory (0: nothing to report), and zeroes them when `clear` is nonzero.
 * No counterpart in the paper: it reports conditions that a kernel records
 * instead of trapping.  The only one in the product build is
 * RLCA_STATUS_WAIT_TIMEOUT: a kernel that waits for its own tensor copies
 * (the time-major bulk driver) gives up after 0.2 s instead of hanging and
 * leaves that call's outputs incomplete.  The copies are synchronous: the
 * call waits for the device's earlier work.  Errors: RLCA_ERR_INVALID_ARG
 * for a NULL `status`, RLCA_ERR_CUDA when a copy fails.
 */
int rlca_device_status(unsigned int *status, int clear);

/* 1 in the index-check build of this library (compiled with
 * RLCA_INDEX_CHECK: kernels check every index of the staged and two-pass
 * paths, record a miss as RLCA_STATUS_INDEX instead of trapping, and each
 * call waits for its kernels, returning RLCA_ERR_CUDA if any recorded a
 * condition), 0 in the product build.  A debugging aid; no counterpart in
 * the paper. */
int rlca_index_checks(void);

/*
 * Bytes of device workspace that the call of `estimator` (RLCA_EST_*) with
 * these sizes and flags needs on the CURRENT device (0 for the one-pass
 * path).  num_actions is read for RLCA_EST_RETRACE only.  Writes the size to
 * *bytes.  Errors: RLCA_ERR_INVALID_ARG for a NULL `bytes`, an unknown
 * estimator, bad sizes or flags; RLCA_ERR_CUDA if the device cannot be
 * queried.
 */
int rlca_workspace_size(int estimator, int64_t E, int64_t T,
                        int32_t num_actions, uint32_t flags, size_t *bytes);

/*
 * Generalized Advantage Estimation (rl-triton §2.1 Motivation, §3.2;
 * Schulman et al. 2016), backward scan with the bootstrap in alpha_{T-1}:
 *   delta_t = r_t + gamma * V_next(t) - V_t
 *   adv_t   = delta_t + gamma * lambda * (1 - d_t) * [t < T-1] * adv_{t+1}
 *   ret_t   = adv_t + V_t
 * V_next(t) = 0 / trunc_value[t] / bootstrap / values[t+1] per the boundary
 * rules above.
 *   rewards, values        [E,T] f32, required
 *   terminated             [E,T] u8, NULL = no terminations
 *   truncated              [E,T] u8, NULL = no truncations (fast path)
 *   trunc_value            [E,T] f32, required iff truncated != NULL; read
 *                          only where truncated is set
 *   bootstrap              [E] f32, NULL = 0
 *   advantages             [E,T] f32 output, required
 *   returns                [E,T] f32 output, NULL = not written
 */
int rlca_gae(const float *rewards, const float *values,
             const uint8_t *terminated, const uint8_t *truncated,
             const float *trunc_value, const float *bootstrap,
             float *advantages, float *returns,
             int64_t E, int64_t T, float gamma, float lambda,
             uint32_t flags, void *workspace, size_t workspace_bytes,
             rlca_stream_t stream);

/*
 * Fused value targets: GAE advantages and returns, discounted returns and
 * TD(lambda) returns of the same rollout in one pass that reads rewards,
 * values and flags once (rl-triton §4 Fusion: constructing coefficients on
 * chip removes intermediate HBM round trips).  The recurrences of rlca_gae
 * and rlca_discounted_return are scanned side by side; the TD(lambda) return
 * is written as advantages + values, which equals it exactly under every
 * boundary rule, so it needs no third scan.  Results equal those of the
 * separate calls within floating-point rounding.
 *   rewards, values, terminated, truncated, trunc_value, bootstrap  as rlca_gae
 *   advantages, returns        [E,T] f32 outputs of rlca_gae, each nullable
 *   disc_returns               [E,T] f32 output of rlca_discounted_return, nullable
 *   td_lambda_returns          [E,T] f32 output of rlca_td_lambda, nullable
 * At least one output must be given.  Workspace (two-pass path): 16 bytes
 * per row per segment (rlca_workspace_size with RLCA_EST_VALUE_TARGETS).
 */
int rlca_value_targets(const float *rewards, const float *values,
                       const uint8_t *terminated, const uint8_t *truncated,
                       const float *trunc_value, const float *bootstrap,
                       float *advantages, float *returns, float *disc_returns,
                       float *td_lambda_returns, int64_t E, int64_t T,
                       float gamma, float lambda, uint32_t flags,
                       void *workspace, size_t workspace_bytes,
                       rlca_stream_t stream);

/*
 * GAE with library-owned scratch, for callers that cannot allocate.
 *
 * The paper has no counterpart to this entry point.  It computes exactly
 * what rlca_gae computes, with the same arguments minus the workspace, for
 * callers that have no way to hand this library a device buffer: a plain C
 * or Fortran host linked only against this library, a simulator callback
 * that must not touch the device heap, a service that reserved all device
 * memory at start-up.  When the two-pass path needs scratch, it uses one
 * array that the library defines in device memory: RLCA_STATIC_SCRATCH_BYTES
 * (1 MiB) on every GPU that loads the library, held until the process exits.
 * Nothing is allocated, on the host or the device, by this call.
 *
 *  - The first call on a device looks up that array's device address (the
 *    set-up); make that first call before any stream capture on the device.
 *    The address is kept with the id of the device context it was found in
 *    and looked up again when that context has changed (after
 *    cudaDeviceReset, for instance): the first call after such a change is
 *    a set-up call too.
 *  - Problems whose two-pass path needs more than RLCA_STATIC_SCRATCH_BYTES
 *    (8 bytes per row per segment; rlca_workspace_size with RLCA_EST_GAE
 *    gives the figure) return RLCA_ERR_UNSUPPORTED and enqueue nothing;
 *    use rlca_gae with a workspace for those.
 *  - All calls on a device share the array and it keeps whatever the last
 *    call left there.  No slot needs to start at zero: the first pass writes
 *    every slot the second pass reads.  Calls whose work overlaps on the GPU
 *    (other streams, other host threads) race on the array and give wrong
 *    results: serialise them.
 * Flags: RLCA_TIME_MAJOR and RLCA_MULTIPASS (RLCA_INPUTS_READY and other
 * bits: RLCA_ERR_INVALID_ARG; RLCA_BF16: RLCA_ERR_UNSUPPORTED).  Arguments,
 * layouts and errors otherwise as rlca_gae.
 */
#define RLCA_STATIC_SCRATCH_BYTES (1u << 20)

int rlca_gae_static_scratch(const float *rewards, const float *values,
                            const uint8_t *terminated,
                            const uint8_t *truncated,
                            const float *trunc_value, const float *bootstrap,
                            float *advantages, float *returns, int64_t E,
                            int64_t T, float gamma, float lambda,
                            uint32_t flags, rlca_stream_t stream);

/*
 * Discounted return (rl-triton §3.2: continuation split between the local
 * update and the boundary carry):
 *   G_t = r_t + gamma * G_next(t),  G_next = 0 / trunc_value[t] /
 *   bootstrap (t = T-1) / G_{t+1}.
 * Scan form: alpha_t = r_t + gamma * trunc_t * trunc_value_t,
 * beta_t = gamma * (1 - d_t), carry A_T = bootstrap.
 * Arguments as rlca_gae; `returns` [E,T] f32 output, required.
 */
int rlca_discounted_return(const float *rewards, const uint8_t *terminated,
                           const uint8_t *truncated, const float *trunc_value,
                           const float *bootstrap, float *returns,
                           int64_t E, int64_t T, float gamma,
                           uint32_t flags, void *workspace,
                           size_t workspace_bytes, rlca_stream_t stream);

/*
 * TD(lambda) return (rl-triton §3.2: continuation split between alpha and
 * the boundary carry):
 *   G_t = r_t + gamma * [(1 - lambda) * V_{t+1} + lambda * G_{t+1}]
 * inside an episode, the bracket replaced by the boundary value at an edge
 * (at t = T-1: (1-lambda)*gamma*bootstrap in alpha, lambda*gamma*bootstrap
 * through the carry A_T = bootstrap).  Arguments as rlca_gae; `returns`
 * [E,T] f32 output, required.
 */
int rlca_td_lambda(const float *rewards, const float *values,
                   const uint8_t *terminated, const uint8_t *truncated,
                   const float *trunc_value, const float *bootstrap,
                   float *returns, int64_t E, int64_t T, float gamma,
                   float lambda, uint32_t flags, void *workspace,
                   size_t workspace_bytes, rlca_stream_t stream);

/*
 * V-Trace (rl-triton §8 Related Work; Espeholt et al. 2018), backward scan
 * with the bootstrap in alpha_{T-1}:
 *   ratio_t = exp(logp_target_t - logp_behaviour_t)
 *   rho_t = min(rho_bar, ratio_t),  c_t = lambda * min(c_bar, ratio_t)
 *   D_t   = rho_t (r_t + gamma V_next(t) - V_t) + gamma c_t (1-d_t)[t<T-1] D_{t+1}
 *   vs_t  = V_t + D_t
 *   pg_t  = rho_t (r_t + gamma vs_next(t) - V_t)   (vs_next: vs_{t+1} inside
 *                                                   an episode, boundary
 *                                                   value at an edge)
 *   logp_target, logp_behaviour  [E,T] f32 log-probabilities of the taken
 *                                action, required
 *   vs                           [E,T] f32 output, required
 *   pg_advantages                [E,T] f32 output, NULL = not written
 * Other arguments as rlca_gae (lambda = 1 gives plain V-Trace).
 */
int rlca_vtrace(const float *rewards, const float *values,
                const float *logp_target, const float *logp_behaviour,
                const uint8_t *terminated, const uint8_t *truncated,
                const float *trunc_value, const float *bootstrap,
                float *vs, float *pg_advantages,
                int64_t E, int64_t T, float gamma, float rho_bar,
                float c_bar, float lambda, uint32_t flags, void *workspace,
                size_t workspace_bytes, rlca_stream_t stream);

/*
 * Retrace(lambda) (rl-triton §3.3: the decay sits on the next step's
 * importance weight; Munos et al. 2016), backward scan with the bootstrap in
 * alpha_{T-1}:
 *   EV_t = sum_a pi[t,a] Q[t,a],  c_t = lambda * min(1, pi[t,a_t] / mu_a[t])
 *   G_t  = r_t + gamma [EV_{t+1} + c_{t+1} (G_{t+1} - Q[t+1, a_{t+1}])]
 * inside an episode, the bracket replaced by the boundary value at an edge
 * (trunc_value: E_pi Q of the truncated episode's last state; bootstrap:
 * E_pi Q of the state after the window).  The action dimension is reduced
 * per step on chip before the scan, so registers do not grow with T.
 *   q, pi        [E,T,A] f32, or bf16 with RLCA_BF16 (A = num_actions
 *                fastest), required
 *   mu_a         [E,T] f32 (bf16 with RLCA_BF16) behaviour probability of
 *                the taken action (> 0)
 *   actions      [E,T] int32 in [0, A); values outside are clamped into
 *                range (memory-safe, result unspecified)
 *   q_ret        [E,T] f32 output, required
 *   num_actions  1 .. RLCA_MAX_ACTIONS (larger: RLCA_ERR_UNSUPPORTED)
 */
int rlca_retrace(const float *q, const float *pi, const float *mu_a,
                 const int32_t *actions, const float *rewards,
                 const uint8_t *terminated, const uint8_t *truncated,
                 const float *trunc_value, const float *bootstrap,
                 float *q_ret, int64_t E, int64_t T, int32_t num_actions,
                 float gamma, float lambda, uint32_t flags, void *workspace,
                 size_t workspace_bytes, rlca_stream_t stream);

/*
 * Accumulating eligibility trace, forward scan (rl-triton §1 forward-time
 * mirror; §5 forward-scan boundaries: beta_t = 0 when d_{t-1} = 1):
 *   e_t = x_t + gamma * lambda * (1 - d_{t-1}) * e_{t-1},  e_{-1} = 0.
 *   x           [E,T] f32 per-step signal, required
 *   terminated  [E,T] u8, NULL = none;  truncated [E,T] u8, NULL = none
 *   out         [E,T] f32 output, required
 */
int rlca_elig_trace(const float *x, const uint8_t *terminated,
                    const uint8_t *truncated, float *out, int64_t E,
                    int64_t T, float gamma, float lambda, uint32_t flags,
                    void *workspace, size_t workspace_bytes,
                    rlca_stream_t stream);

/*
 * Episodic prefix sum, segmented forward scan (rl-triton §3.3: configurable
 * boundary conventions):
 *   S_t = x_t + (1 - d_{t-1}) S_{t-1}       (default, flag = last step)
 *   S_t = x_t + (1 - d_t) S_{t-1}           (RLCA_PSUM_FLAG_IS_START)
 * RLCA_PSUM_EXCLUSIVE writes S_t - x_t (the sum over the earlier steps of t's
 * episode).  d = terminated | truncated (either may be NULL).
 *   x, out  [E,T] of `dtype`: RLCA_I32 (int32, wraps modulo 2^32,
 *           bit-exact) or RLCA_F32 (float32)
 */
int rlca_episodic_prefix_sum(const void *x, int dtype,
                             const uint8_t *terminated,
                             const uint8_t *truncated, void *out,
                             int64_t E, int64_t T, uint32_t flags,
                             void *workspace, size_t workspace_bytes,
                             rlca_stream_t stream);

/*
 * Generic affine scan over precomputed coefficients (rl-triton §4 Scan
 * procedure: the generic kernel consuming precomputed alpha and beta).
 *   reverse != 0: A_t = alpha_t + beta_t A_{t+1}, A_T    = carry[e]
 *   reverse == 0: A_t = alpha_t + beta_t A_{t-1}, A_{-1} = carry[e]
 *   alpha, beta  [E,T] f32, required;  carry [E] f32, NULL = 0
 *   out          [E,T] f32 output, required
 */
int rlca_affine_scan(const float *alpha, const float *beta,
                     const float *carry, float *out, int64_t E, int64_t T,
                     int reverse, uint32_t flags, void *workspace,
                     size_t workspace_bytes, rlca_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RLCA_H */
