"""GPU parity: every estimator through the C ABI against the float64 oracle.

Workloads follow the benchmark configurations of the rl-triton paper's
massively parallel regime: the 8 x 16 GAE case, 4096 x 128 (GAE, discounted
return, TD(lambda)), 4096 x 256 V-Trace, 1024 x 2048 Retrace with 18 actions,
and the sweep of all estimators over E in {256, 1024, 4096, 16384} x
T in {32, 128, 512, 2048}, both layouts, with and without truncation; plus
edge cases (T = 1, ragged T, tile +- 1, E = 1, misaligned pointers, the
two-pass path, both flags on one step, int32 wraparound).
"""
import ctypes as C

import numpy as np
import pytest
import torch

from first_order_linear_gb300 import _lib, rlca, synth
from tests import parity

pytestmark = pytest.mark.gpu

ESTIMATORS = ["gae", "disc", "td", "vtrace", "retrace", "elig", "psum_i32"]
SWEEP = ESTIMATORS + ["vt"]


@pytest.fixture(autouse=True)
def _gpu(cuda_lib):
    yield


# --------------------------------------------------------------------------
# the named workloads
# --------------------------------------------------------------------------

def test_gae_8x16_seed0():
    """GAE fp32, 8 envs x 16 steps, seed 0, termination 5%, truncation 2%."""
    d = synth.value_rollout(8, 16, seed=0, p_term=0.05, p_trunc=0.02, with_trunc=True)
    for tm in (False, True):
        for mp in (False, True):
            parity.check_case("gae", 8, 16, inputs=d, time_major=tm, multipass=mp)


@pytest.mark.parametrize("kind", ["gae", "disc", "td", "vt"])
@pytest.mark.parametrize("trunc", [True, False])
def test_4096x128_value_estimators(kind, trunc):
    d = synth.value_rollout(4096, 128, seed=synth.config_seed("4096x128"), p_term=0.01, p_trunc=0.005,
                            with_trunc=trunc)
    parity.check_case(kind, 4096, 128, inputs=d, rows=np.arange(4096))


def test_vtrace_4096x256():
    d = synth.vtrace_rollout(4096, 256, seed=synth.config_seed("vtrace4096x256"), p_term=0.01)
    parity.check_case("vtrace", 4096, 256, inputs=d, rows=np.arange(4096))


def test_retrace_1024x2048():
    d = synth.retrace_rollout(1024, 2048, seed=synth.config_seed("retrace1024x2048"), p_term=0.002,
                              device="cuda")
    parity.check_case("retrace", 1024, 2048, inputs=d, rows=np.arange(1024))


@pytest.mark.parametrize("trunc", [False, True], ids=["notrunc", "trunc"])
@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
@pytest.mark.parametrize("T", [32, 128, 512, 2048])
@pytest.mark.parametrize("E", [256, 1024, 4096, 16384])
@pytest.mark.parametrize("kind", SWEEP)
def test_sweep(kind, E, T, tm, trunc):
    seed = synth.config_seed(f"sweep-{kind}-{E}-{T}-{tm}-{trunc}")
    parity.check_case(kind, E, T, seed=seed, trunc=trunc, time_major=tm, gen_device="cuda")


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------

EDGE_T = [1, 2, 3, 4, 5, 7, 15, 16, 17, 31, 33, 63, 65, 127, 129, 255, 257, 1023, 1025, 2047, 2049, 4095,
          4097, 8193]


@pytest.mark.parametrize("kind", parity.KINDS)
@pytest.mark.parametrize("T", EDGE_T)
def test_ragged_lengths(kind, T):
    for E, tm, mp in ((3, False, False), (33, True, False), (5, False, True), (2, True, True)):
        parity.check_case(kind, E, T, seed=T * 7 + E, trunc=True, time_major=tm, multipass=mp, p_term=0.05)


@pytest.mark.parametrize("kind", parity.KINDS)
def test_single_env_and_dense_boundaries(kind):
    parity.check_case(kind, 1, 300, seed=1, p_term=0.0)
    parity.check_case(kind, 7, 64, seed=2, p_term=0.5)
    parity.check_case(kind, 7, 64, seed=3, p_term=1.0)


@pytest.mark.parametrize("kind", ["gae", "disc", "td", "vt", "vtrace", "retrace", "elig", "psum_f32",
                                  "affine_bwd"])
@pytest.mark.parametrize("tm", [False, True])
def test_long_rows_few_envs_two_pass(kind, tm):
    """Rows much longer than one tile on a handful of environments take the
    segmented two-pass path by themselves."""
    parity.check_case(kind, 3, 40000, seed=11, time_major=tm)


@pytest.mark.parametrize("kind", ["gae", "vt", "retrace", "elig", "psum_i32", "affine_fwd"])
@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
def test_rows_beyond_131072_steps(kind, tm):
    """Rows longer than the 131072-step limit of the pages' fused kernels
    (their backward-only unfused fallback beyond it) run the segmented
    two-pass path, backward and forward alike."""
    parity.check_case(kind, 2, 140_001, seed=17, time_major=tm, p_term=0.0005)


@pytest.mark.parametrize("kind", parity.KINDS)
@pytest.mark.parametrize("T", [8, 16, 24, 32, 64, 128, 256, 520, 2048])
def test_time_major_chunk_groups(kind, T):
    """Time-major rows of whole 8-step chunks run the fast time-major drivers
    (direct or staged): 8 environments per CTA below 64 x SMs environments,
    32 from there on, with 1 to 32 chunk lanes per environment; ragged E on
    both sides."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 32 environments per CTA and E % 4 == 0 stream through shared-memory stages; the rest read
    # straight into registers
    for E, seed in ((13, 1), (12, 2), (64 * sms + 5, 3), (64 * sms + 4, 4)):
        parity.check_case(kind, E, T, seed=T * 11 + seed, time_major=True, p_term=0.02)
    for E, seed in ((13, 5), (12, 6)):
        parity.check_case(kind, E, T, seed=T * 11 + seed, time_major=True, p_term=0.02, inputs_ready=True)


@pytest.mark.parametrize("kind", [k for k in parity.KINDS if k != "retrace"])
@pytest.mark.parametrize("E,T", [(5, 40000), (12, 8192), (300, 4096), (1023, 2048)])
def test_time_major_two_pass_fast_drivers(kind, E, T):
    """Few environments with long whole-chunk rows, time-major: the fast and
    staged time-major drivers run the two-pass split (segment maps, then the
    segments from their entering values); direct (E % 4 != 0) and staged
    tiles, both stream modes."""
    parity.check_case(kind, E, T, seed=E + T, time_major=True, p_term=0.005)
    parity.check_case(kind, E, T, seed=E + T + 1, time_major=True, p_term=0.005, inputs_ready=True)


@pytest.mark.parametrize("kind", parity.KINDS)
@pytest.mark.parametrize("T", [16, 64, 256, 1024])
def test_more_row_groups_than_one_wave(kind, T):
    """Single-tile env-major calls with many waves of CTAs (hundreds of
    thousands of rows, ragged E), in both stream modes."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    E = 40 * sms * 4096 // max(T, 64) + 5
    parity.check_case(kind, E, T, seed=T + 31, p_term=0.02)
    parity.check_case(kind, E, T, seed=T + 32, p_term=0.02, inputs_ready=True)


@pytest.mark.parametrize("kind", parity.KINDS)
@pytest.mark.parametrize("T", [256, 512])
def test_mid_rows_eight_steps_a_thread(kind, T):
    """Rows of 256-1023 steps on environments that fill the GPU twice over
    take 8 steps a thread (one or two warps a row), ragged E."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    E = -(-2 * sms * 1024 // (T // 8)) + 3
    parity.check_case(kind, E, T, seed=T + 41, p_term=0.02)
    parity.check_case(kind, E, T, seed=T + 42, p_term=0.02, inputs_ready=True)


@pytest.mark.parametrize("kind", parity.KINDS)
@pytest.mark.parametrize("T", [1024, 3072, 4096])
def test_long_single_tile_rows(kind, T):
    """Rows of 1024-4096 steps fit one tile.  With few environments the fast
    env-major driver runs them with 4 steps per thread; once E*T/8 threads
    fill the GPU (four times that for Retrace) with 8 steps per thread.  Both
    sides of that switch are checked, with a ragged environment count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = sms * 1024 * (4 if kind == "retrace" else 1)
    e_long = -(-need // (T // 8)) + 3
    parity.check_case(kind, 70, T, seed=T + 3, p_term=0.01)
    parity.check_case(kind, e_long, T, seed=T + 4, p_term=0.01)
    parity.check_case(kind, e_long, T, seed=T + 5, p_term=0.01, inputs_ready=True)


@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
@pytest.mark.parametrize("kind", parity.KINDS)
def test_misaligned_pointers(kind, tm):
    """Inputs at 4-byte (flags: 1-byte) rather than 16-byte offsets take the
    unstaged scalar load paths and must give the same results; E = 36 and
    T = 96 would otherwise take the vector / staged paths."""
    parity.check_case(kind, 36, 96, seed=5, p_term=0.05, time_major=tm, shift=True)
    parity.check_case(kind, 37, 96, seed=6, p_term=0.05, time_major=tm, shift=True)


@pytest.mark.parametrize("kind", ["gae", "disc", "td", "vt", "vtrace", "retrace"])
def test_termination_wins_over_truncation(kind):
    E, T = 16, 50
    d = parity.make_inputs(kind, E, T, seed=9, trunc=True, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9)
    both = torch.rand(E, T, generator=g, device="cuda") < 0.2
    d["terminated"] = (d["terminated"].bool() | both).to(torch.uint8)
    d["truncated"] = (d["truncated"].bool() | both).to(torch.uint8)
    if d.get("trunc_value") is None:
        d["trunc_value"] = torch.randn(E, T, generator=g, device="cuda")
    parity.check_case(kind, E, T, inputs=d)
    parity.check_case(kind, E, T, inputs=d, time_major=True)


@pytest.mark.parametrize("exclusive", [False, True])
@pytest.mark.parametrize("flag_is_start", [False, True])
@pytest.mark.parametrize("kind", ["psum_i32", "psum_f32"])
def test_prefix_sum_conventions(kind, exclusive, flag_is_start):
    p = dict(exclusive=exclusive, flag_is_start=flag_is_start)
    for E, T, tm, mp in ((64, 200, False, False), (64, 200, True, False), (5, 777, False, True),
                         (9, 131, True, True)):
        parity.check_case(kind, E, T, seed=E + T, time_major=tm, multipass=mp, params=p, p_term=0.05)


def test_prefix_sum_int32_wraps():
    E, T = 4, 1000
    x = torch.full((E, T), 2 ** 30 + 12345, dtype=torch.int32, device="cuda")
    x[1] = -(2 ** 31) + 7
    term = torch.zeros(E, T, dtype=torch.uint8, device="cuda")
    term[2, 500] = 1
    d = dict(x_i32=x, x_f32=x.float(), terminated=term, truncated=None)
    for tm in (False, True):
        parity.check_case("psum_i32", E, T, inputs=d, time_major=tm)


@pytest.mark.parametrize("A", [1, 2, 5, 18, 33, 64])
def test_retrace_action_counts(A):
    for tm in (False, True):
        parity.check_case("retrace", 24, 160, seed=A, time_major=tm, num_actions=A, p_term=0.02)


def test_retrace_time_major_widths():
    """Time-major Retrace at each staging width: 16 chunk warps (128-step
    tiles) where the environments give at most one CTA per SM, 8 beyond
    that, 8 with two-pass segments for few environments with long rows,
    and fewer where many actions fill the staging buffers; float32 and
    bfloat16."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [(32 * sms, 512, 18), (32 * sms + 32, 256, 18), (1024, 1024, 18), (32 * sms, 256, 64)]
    for i, (E, T, A) in enumerate(cases):
        for bf16 in (False, True):
            parity.check_case("retrace", E, T, seed=70 + i, time_major=True, num_actions=A, bf16=bf16)


@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("E,T", [(13, 2048), (256, 2048), (1000, 1000), (1001, 1003), (40, 4096), (8, 72)])
def test_retrace_time_major_second_pass(E, T, bf16):
    """Time-major Retrace on few environments splits rows into segments; the
    second pass scans the per-step scalars the first left in the workspace
    on the fast time-major driver (CTAs of 8 environments, 16 for bfloat16,
    1 to 32 chunk threads to fit the segment) when T % 8 == 0, and with the
    first pass's kernel otherwise (T = 1003).  Ragged E, truncation on, also
    with termination everywhere in some rows."""
    parity.check_case("retrace", E, T, seed=E + T, time_major=True, bf16=bf16, p_term=0.002)
    parity.check_case("retrace", E, T, seed=E + T + 1, time_major=True, bf16=bf16, p_term=0.3)


def test_vtrace_clipping_and_lambda():
    p = dict(rho_bar=1.3, c_bar=0.7, vt_lambda=0.9)
    for tm in (False, True):
        parity.check_case("vtrace", 300, 96, seed=4, time_major=tm, params=p)


def test_gamma_lambda_extremes():
    for g, lam in ((0.0, 0.0), (1.0, 1.0), (0.5, 0.0), (1.0, 0.0)):
        p = dict(gamma=g, lambda_=lam)
        for kind in ("gae", "disc", "td", "vt", "elig"):
            parity.check_case(kind, 50, 70, seed=8, params=p)


# --------------------------------------------------------------------------
# properties at full size
# --------------------------------------------------------------------------

def test_layouts_agree_full_size():
    E, T = 4096, 512
    for kind in ESTIMATORS:
        d = parity.make_inputs(kind, E, T, seed=77, trunc=True, device="cuda")
        a = parity.run_gpu(kind, d, time_major=False)
        b = parity.run_gpu(kind, d, time_major=True)
        for x, y in zip(a, b):
            if x is None:
                continue
            if x.dtype == torch.int32:
                assert torch.equal(x, y), kind
            else:
                err = ((x.double() - y.double()).abs() / (1 + y.double().abs())).max().item()
                assert err <= 2 * parity.TOL, (kind, err)


def test_fused_value_targets_match_separate_calls_full_size():
    d = parity.make_inputs("gae", 16384, 2048, seed=80, trunc=True, device="cuda")
    fused = parity.run_gpu("vt", d)
    sep = parity.run_gpu("gae", d) + parity.run_gpu("disc", d) + parity.run_gpu("td", d)
    for a, b in zip(fused, sep):
        err = ((a.double() - b.double()).abs() / (1 + b.double().abs())).max().item()
        assert err <= 2 * parity.TOL


def test_td_lambda_equals_gae_returns_full_size():
    d = parity.make_inputs("gae", 16384, 2048, seed=78, trunc=True, device="cuda")
    adv, ret = parity.run_gpu("gae", d)
    (td,) = parity.run_gpu("td", d)
    err = ((td.double() - ret.double()).abs() / (1 + ret.double().abs())).max().item()
    assert err <= 2 * parity.TOL


def test_deterministic_and_stream_ordered():
    d = parity.make_inputs("gae", 4096, 128, seed=79, trunc=True, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        a = parity.run_gpu("gae", d)
    s.synchronize()
    b = parity.run_gpu("gae", d)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("kind", parity.KINDS)
def test_inputs_ready_flag_gives_the_same_results(kind):
    """RLCA_INPUTS_READY only changes when a kernel may start reading."""
    for E, T, tm in ((4096, 128, False), (300, 1000, True), (7, 9000, False)):
        parity.check_case(kind, E, T, seed=E + T, time_major=tm, inputs_ready=True)


def test_inputs_ready_chain_keeps_stream_order():
    """Back-to-back calls in one stream: calls flagged RLCA_INPUTS_READY
    overlap their predecessor, while an unflagged call that reads the
    previous call's output still sees it complete.  Each affine scan feeds
    the next one's alpha; the final result must match running them one by
    one with a synchronisation in between."""
    E, T = 4096, 512
    d = parity.make_inputs("affine_bwd", E, T, seed=91, trunc=False, device="cuda")
    beta = d["beta"] * 0.5
    indep = [torch.randn(E, T, device="cuda") for _ in range(6)]
    torch.cuda.synchronize()
    outs = []
    cur = d["alpha"]
    for i in range(6):
        # unflagged: reads the previous result
        cur = rlca.rlca_affine_scan(cur * 0 + cur, beta, None)  # copy kernel in between, then scan
        cur = rlca.rlca_affine_scan(cur, beta, None)
        # flagged calls on independent inputs interleaved
        outs.append(rlca.rlca_affine_scan(indep[i], beta, None, inputs_ready=True))
        cur = rlca.rlca_affine_scan(cur, beta, None)
    torch.cuda.synchronize()
    ref_cur = d["alpha"]
    for i in range(6):
        ref_cur = rlca.rlca_affine_scan(ref_cur * 0 + ref_cur, beta, None)
        torch.cuda.synchronize()
        ref_cur = rlca.rlca_affine_scan(ref_cur, beta, None)
        torch.cuda.synchronize()
        ref_i = rlca.rlca_affine_scan(indep[i], beta, None)
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref_i)
        ref_cur = rlca.rlca_affine_scan(ref_cur, beta, None)
        torch.cuda.synchronize()
    assert torch.equal(cur, ref_cur)


def test_empty_inputs():
    z = torch.empty(0, 16, device="cuda")
    adv, ret = rlca.rlca_gae(z, z.clone())
    assert adv.shape == (0, 16)
    z2 = torch.empty(5, 0, device="cuda")
    assert rlca.rlca_discounted_return(z2).shape == (5, 0)


# --------------------------------------------------------------------------
# large sizes: 64-bit offsets and very long rows (against the C reference,
# which walks long rows quickly; a few sampled rows of the wide cases)
# --------------------------------------------------------------------------

def _big_flags(shape, p, gen):
    return (torch.rand(shape, device="cuda", dtype=torch.float16, generator=gen) < p).to(torch.uint8)


def _check_rows(got, want, what):
    parity.assert_close(got, want, what)


@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
def test_element_offsets_beyond_32_bits(tm):
    """E * T past 2^31 (env-major) and past 2^32 (time-major: the 32-bit
    offset drivers step aside for the general ones): discounted returns and
    eligibility traces on sampled environments.  About 40 GB on the device."""
    from oracle import ref_c
    gen = torch.Generator(device="cuda").manual_seed(99)
    E, T = (65539, 32771) if not tm else (131075, 32771)
    shape = (T, E) if tm else (E, T)
    r = torch.randn(shape, device="cuda", generator=gen)
    term = _big_flags(shape, 0.001, gen)
    rows = np.array([0, 1, E // 2, E - 1])
    pick = (lambda t: t[:, torch.as_tensor(rows, device="cuda")].T) if tm else \
        (lambda t: t[torch.as_tensor(rows, device="cuda")])
    r_s, term_s = pick(r).double().cpu().numpy(), pick(term).cpu().numpy()
    out = rlca.rlca_discounted_return(r, term, time_major=tm)
    torch.cuda.synchronize()
    _check_rows(pick(out).double().cpu().numpy(), ref_c.discounted_return(r_s, term_s, gamma=parity.GAMMA),
                f"disc E={E} T={T} tm={tm}")
    del out
    out = rlca.rlca_elig_trace(r, term, time_major=tm)
    torch.cuda.synchronize()
    _check_rows(pick(out).double().cpu().numpy(),
                ref_c.eligibility_trace(r_s, term_s, gamma=parity.GAMMA, lam=parity.LAMBDA),
                f"elig E={E} T={T} tm={tm}")
    del out, r, term
    torch.cuda.empty_cache()


def test_rows_of_a_hundred_million_steps():
    """T = 2^27 + 5 on two environments: the segmented two-pass path (each
    segment hundreds of tiles long, unaligned row ends), backward and
    forward."""
    from oracle import ref_c
    gen = torch.Generator(device="cuda").manual_seed(7)
    E, T = 2, (1 << 27) + 5
    r = torch.randn(E, T, device="cuda", generator=gen)
    term = _big_flags((E, T), 1e-6, gen)
    r_h, term_h = r.double().cpu().numpy(), term.cpu().numpy()
    out = rlca.rlca_discounted_return(r, term)
    torch.cuda.synchronize()
    _check_rows(out.double().cpu().numpy(), ref_c.discounted_return(r_h, term_h, gamma=parity.GAMMA), "disc")
    out = rlca.rlca_elig_trace(r, term)
    torch.cuda.synchronize()
    _check_rows(out.double().cpu().numpy(),
                ref_c.eligibility_trace(r_h, term_h, gamma=parity.GAMMA, lam=parity.LAMBDA), "elig")
    del out, r, term
    torch.cuda.empty_cache()


def test_workspace_sizes_consistent():
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, 4096, 128) == 0
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, 3, 40000) > 0
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, 64, 512, flags=_lib.RLCA_MULTIPASS) > 0
    assert rlca.rlca_workspace_size(_lib.RLCA_EST_VALUE_TARGETS, 3, 40000) == \
        2 * rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, 3, 40000)
    d = parity.make_inputs("gae", 3, 40000, seed=1, trunc=False, device="cuda")
    with pytest.raises(ValueError):
        rlca.rlca_gae(d["rewards"], d["values"], workspace=torch.empty(8, dtype=torch.uint8, device="cuda"))


# --------------------------------------------------------------------------
# bfloat16 storage (RLCA_BF16): float32 arithmetic, outputs rounded once
# --------------------------------------------------------------------------

BF16_KINDS = ["gae", "vt", "disc", "td", "vtrace", "retrace", "elig", "psum_f32", "affine_bwd", "affine_fwd"]


@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
@pytest.mark.parametrize("E,T", [(8, 16), (37, 129), (256, 128), (70, 1024), (5, 2048), (3, 40001)])
@pytest.mark.parametrize("kind", BF16_KINDS)
def test_bf16_storage(kind, E, T, tm):
    """bfloat16 inputs and outputs through every driver: the fast drivers
    (whole 4- or 8-step chunks), ragged T (scalar loads), one-tile and
    multi-tile rows and the two-pass segments; against the oracle on the
    same bfloat16 inputs within the rounding bound of parity.BF16_REL."""
    parity.check_case(kind, E, T, seed=E * 131 + T, time_major=tm, bf16=True, p_term=0.02)


@pytest.mark.parametrize("kind", BF16_KINDS)
def test_bf16_wide_time_major_and_modes(kind):
    """The staged time-major driver in bfloat16 (16-byte pieces of 8
    environments: E % 8 == 0), its direct sibling (E % 8 != 0), the
    inputs-ready and two-pass modes, and unaligned bfloat16 inputs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for E, seed in ((64 * sms + 8, 1), (64 * sms + 4, 2)):
        parity.check_case(kind, E, 512, seed=seed, time_major=True, bf16=True, p_term=0.02)
    parity.check_case(kind, 64 * sms + 8, 64, seed=3, time_major=True, bf16=True, inputs_ready=True)
    parity.check_case(kind, 300, 256, seed=4, bf16=True, inputs_ready=True)
    parity.check_case(kind, 6, 3000, seed=5, bf16=True, multipass=True)
    parity.check_case(kind, 6, 3000, seed=6, bf16=True, multipass=True, time_major=True)
    parity.check_case(kind, 36, 96, seed=7, bf16=True, shift=True)
    parity.check_case(kind, 36, 96, seed=8, bf16=True, shift=True, time_major=True)


def test_bf16_value_targets_4096x128():
    """The fused value targets of the 4096 x 128 configuration in bfloat16."""
    parity.check_case("vt", 4096, 128, seed=11, bf16=True)
    parity.check_case("vt", 4096, 128, seed=12, bf16=True, inputs_ready=True)


@pytest.mark.parametrize("A", [1, 3, 18, 64])
@pytest.mark.parametrize("tm", [False, True], ids=["env", "time"])
def test_bf16_retrace_action_counts(A, tm):
    """bfloat16 Q and pi blocks of every parity of A: odd A leaves the
    per-step blocks 2-byte aligned (4-byte and plain-load copies), A = 64
    the 16-byte pieces."""
    parity.check_case("retrace", 40, 200, seed=A, time_major=tm, bf16=True, num_actions=A)
    parity.check_case("retrace", 40, 200, seed=A + 1, time_major=tm, bf16=True, num_actions=A, shift=True)



def test_side_stream_two_pass_workspace_survives_reuse():
    """A call on a stream other than the current one, whose workspace and
    outputs the binding allocates: memory the current stream allocates
    right after the call must not alias them while the kernel runs."""
    E, T = 64, 4096  # few environments, long rows: the two-pass path with a workspace
    d = parity.make_inputs("gae", E, T, seed=11, trunc=True, device="cuda")
    need = rlca.rlca_workspace_size(_lib.RLCA_EST_GAE, E, T, 0, _lib.RLCA_MULTIPASS)
    assert need > 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    rounds = []
    for _ in range(4):
        adv, ret = rlca.rlca_gae(d["rewards"], d["values"], d["terminated"], d["truncated"], d["trunc_value"],
                                 d["bootstrap"], gamma=parity.GAMMA, lambda_=parity.LAMBDA, multipass=True,
                                 stream=side)
        # the current stream grabs and scribbles on fresh memory at once
        junk = [torch.full((need // 4 + 1024,), float("nan"), device="cuda") for _ in range(4)]
        del junk
        rounds.append((adv, ret))
    torch.cuda.synchronize()
    want = parity.run_oracle("gae", d, np.arange(E))
    for adv, ret in rounds:
        parity.assert_close(adv.cpu().numpy(), want[0], "adv on a side stream")
        parity.assert_close(ret.cpu().numpy(), want[1], "ret on a side stream")


def test_retrace_two_pass_keeps_per_step_scalars():
    """Retrace on the two-pass path: the workspace holds the segment maps and
    three float planes of per-step (E_pi Q, Q(a), c), 12 bytes a step, which
    the second pass reads instead of Q and pi; results match the oracle in
    both layouts, also when the workspace held other data before."""
    E, T = 1024, 2048
    for tm in (True, False):
        flags = _lib.RLCA_TIME_MAJOR if tm else 0
        need = rlca.rlca_workspace_size(_lib.RLCA_EST_RETRACE, E, T, synth.NUM_ACTIONS, flags)
        if need == 0:
            continue  # this device runs the layout in one pass
        assert need >= 12 * E * T
        d = synth.retrace_rollout(E, T, seed=synth.config_seed("retrace-aux"), p_term=0.002, p_trunc=0.005,
                                  with_trunc=True, device="cuda")
        x = parity._tm(d, tm)
        ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")  # garbage the first pass must overwrite
        out = rlca.rlca_retrace(x["q"], x["pi"], x["mu_a"], x["actions"], x["rewards"], x["terminated"],
                                x["truncated"], x["trunc_value"], x["bootstrap"], gamma=parity.GAMMA,
                                lambda_=parity.LAMBDA, time_major=tm, workspace=ws)
        torch.cuda.synchronize()
        rows = parity.sample_rows(E, T, seed=5, n=128)
        want = parity.run_oracle("retrace", d, rows)
        parity.assert_close(parity._np(parity._back(out, tm), rows), want[0], f"retrace two-pass tm={tm}")


@pytest.mark.parametrize("kind", ["gae", "vt", "vtrace", "disc", "elig", "psum_i32", "affine_fwd"])
@pytest.mark.parametrize("E,T", [(9728, 16), (9744, 64), (10240, 520), (16384, 256)])
def test_time_major_tile_copies_leave_status_clean(cuda_lib, kind, E, T):
    """Time-major calls with many environments (E >= 64 per SM, E % 16 == 0,
    16-byte aligned inputs) move their tiles by tensor copies with bounded
    waits -- 9744 leaves the last CTA's tile half past E, zero-filled; results
    match the oracle and no wait gives up (the device status word stays 0)."""
    st = C.c_uint(0)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    parity.check_case(kind, E, T, seed=E + T, time_major=True)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    assert st.value == 0, f"device status {st.value:#x}"


@pytest.mark.parametrize("kind", ["gae", "vt", "vtrace", "td", "disc", "elig", "psum_i32", "affine_fwd"])
@pytest.mark.parametrize("E,T", [(16, 8), (1024, 520), (2432, 2048), (4096, 1024), (4096, 2056), (9712, 1024),
                                 (4096, 128)])
def test_time_major_narrow_tile_copies(cuda_lib, kind, E, T):
    """Float32 time-major calls below 64 environments per SM with E % 16 ==
    0, aligned inputs, two or more float inputs, rows of four or more tiles
    and E / 8 >= 2 per SM move tiles of 8 environments by tensor copies; the
    flag rows are copied 16 environments wide and each CTA reads its half
    (odd CTAs the upper one).  The other shapes here take the other drivers;
    results match the oracle and the device status word stays 0."""
    st = C.c_uint(0)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    parity.check_case(kind, E, T, seed=E + T + 1, time_major=True, p_term=0.02)
    parity.check_case(kind, E, T, seed=E + T + 2, time_major=True, inputs_ready=True)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    assert st.value == 0, f"device status {st.value:#x}"


@pytest.mark.parametrize("kind", ["gae", "vt", "vtrace", "td", "disc", "elig", "psum_i32", "affine_fwd"])
@pytest.mark.parametrize("E,T", [(8, 64), (1000, 520), (4096, 2048), (256, 4096)])
def test_time_major_few_envs_repeated_calls(cuda_lib, kind, E, T):
    """Time-major calls with few environments and rows of several tiles (the
    direct 8-environment driver, walking tiles; the two-pass split where the
    rows are long and few), two calls in a row, the second's workspace
    memory reused from the first: both match the oracle, with the device
    status word clean."""
    st = C.c_uint(0)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    for call in range(2):
        d = parity.make_inputs(kind, E, T, seed=call * 1000 + E + T, trunc=True, device="cuda")
        parity.check_case(kind, E, T, inputs=d, time_major=True)
    assert cuda_lib.rlca_device_status(C.byref(st), 1) == _lib.RLCA_OK
    assert st.value == 0, f"device status {st.value:#x}"


def test_time_major_bf16_few_envs_workspace_garbage(cuda_lib):
    """bfloat16 storage, time-major with few environments and long rows (16
    environments a CTA), with a caller workspace full of 0xFF bytes before
    each of two calls."""
    E, T = 1024, 2048
    need = rlca.rlca_workspace_size(_lib.RLCA_EST_VALUE_TARGETS, E, T, 0, _lib.RLCA_TIME_MAJOR | _lib.RLCA_BF16)
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    for call in range(2):
        d = parity.to_bf16(parity.make_inputs("vt", E, T, seed=77 + call, trunc=True, device="cuda"))
        ws.fill_(0xFF)
        x = parity._tm(d, True)
        out = rlca.rlca_value_targets(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                                      x["bootstrap"], gamma=parity.GAMMA, lambda_=parity.LAMBDA, time_major=True,
                                      workspace=ws if need > 0 else None)
        torch.cuda.synchronize()
        rows = parity.sample_rows(E, T, seed=call)
        want = parity.run_oracle("vt", d, rows)
        for o, w, name in zip(out[:3], want[:3], ("adv", "ret", "disc")):
            parity.assert_close(parity._np(parity._back(o, True), rows), w, f"bf16 time-major {name} call {call}",
                                tol=parity.BF16_TOL, rel=parity.BF16_REL)
