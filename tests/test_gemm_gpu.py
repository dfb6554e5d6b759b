"""GPU parity of every kernel variant against the CPU oracle, through the C ABI.

* integer-valued operands: every fp32 partial sum is exact, so the GPU must
  match the oracle bit for bit (bf16 output: the oracle's exact integer
  rounded to nearest even);
* random operands: the per-element acceptance rule of oracle.parity;
* ragged shapes that span several tiles in M, N and K;
* the scheduler covers every tile exactly once;
* a forced device-side wait timeout is reported and leaves the context usable.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from dense_gemm_blackwell_sm_gb300 import gemm, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def run_variant(a, b, out, variant, sched=0, stages=0, raster_group=0, max_ctas=0, plan_out=None):
    M, K = a.shape
    N = b.shape[0]
    code = gemm.dtype_code(a.dtype, out)
    plan = gemm.Plan(M, N, K, code, gemm.make_opts(variant=variant, sched=sched, stages=stages,
                                                   raster_group=raster_group, max_ctas=max_ctas))
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(out))
    plan.run(a.to(DEV), b.to(DEV), c)
    st = plan.check()
    assert st == gemm.OK, gemm.status_string(st)
    if plan_out is not None:
        plan_out.append(plan.info())
    plan.destroy()
    return c.float().cpu().numpy().astype(np.float64)


def expect_bits(ref: np.ndarray, out: str) -> np.ndarray:
    """The exact result in the output format (bf16: round to nearest even)."""
    t = torch.tensor(ref, dtype=torch.float64)
    if out == "bf16":
        return t.to(torch.bfloat16).to(torch.float64).numpy()
    return t.to(torch.float32).to(torch.float64).numpy()


# variant -> ragged shapes spanning several of its tiles (N % 8 == 0 throughout)
SHAPES = {
    gemm.S1: [(128, 128, 64), (100, 72, 40)],
    gemm.S2: [(128, 128, 512), (77, 120, 136)],
    gemm.S3: [(300, 264, 520), (129, 8, 72)],
    gemm.S4: [(300, 264, 520)],
    gemm.S5: [(300, 264, 520), (257, 392, 1000)],
    gemm.S6: [(300, 264, 520), (1030, 1288, 264)],
    gemm.S7: [(300, 520, 200), (700, 1288, 264)],
    gemm.S8: [(300, 520, 200), (700, 1288, 264), (1, 264, 72)],
    gemm.S9: [(300, 520, 200), (1100, 1288, 264)],
    # GEMV: the K-split kernel (M <= 2 and at most 64 rows per SM) and the row kernel
    gemm.GEMV: [(1, 1000, 520), (3, 264, 72), (8, 1000, 520), (16, 96, 1024), (1, 4096, 4096), (2, 152, 8),
                # 3 <= M <= 8 with the activations in shared memory: an odd number of load
                # groups per row group (no prefetch across row groups), several row groups
                # per warp (prefetch across them), ragged rows
                (8, 2000, 8200), (4, 20000, 4096), (6, 777, 264),
                (1, 1, 64), (1, 9000, 16384), (2, 777, 4104), (1, 500, 8), (2, 12000, 520),
                # one activation row, K a multiple of 1024: the rolling kernel, with a
                # whole row per load group (K = 1024) and several rows per warp
                (1, 1000, 1024), (1, 20000, 2048)],
    gemm.GEMV_TC: [(1, 1000, 520), (3, 264, 72), (8, 1000, 4104), (16, 96, 1024)],
}
CASES = [(v, s) for v, shapes in SHAPES.items() for s in shapes]
IDS = ["%s-%dx%dx%d" % (gemm.VARIANT_NAMES[v], *s) for v, s in CASES]


@pytest.mark.parametrize("variant,shape", CASES, ids=IDS)
@pytest.mark.parametrize("ti,to", [("f16", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f16", "bf16")])
def test_integer_inputs_bit_exact(variant, shape, ti, to):
    M, N, K = shape
    a, b = inputs.integer_operands(M, N, K, ti, seed=M * 7 + N * 3 + K)
    ref, _ = oracle.gemm(a, b)
    c = run_variant(a, b, to, variant)
    exp = expect_bits(ref, to)
    bad = np.argwhere(c != exp)
    assert bad.size == 0, "first mismatch at %s: got %r expected %r" % (
        bad[0], c[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("variant,shape", [(gemm.S7, (2048, 8192, 264)), (gemm.S8, (2048, 8192, 264)),
                                           (gemm.S9, (4096, 8192, 264))], ids=["s7", "s8", "s9"])
@pytest.mark.parametrize("sched", [gemm.SCHED_STATIC, gemm.SCHED_ATOMIC])
def test_several_tiles_per_cluster_bit_exact(variant, shape, sched):
    """Every cluster takes three or more tiles, so its odd-numbered tiles run
    their K blocks backwards (starting with the ragged last block): the result
    must still be exact."""
    M, N, K = shape
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=41)
    ref, _ = oracle.gemm(a, b)
    info = []
    c = run_variant(a, b, "f32", variant, sched=sched, plan_out=info)
    assert info[0]["tiles"] >= 3 * (info[0]["grid"] // info[0]["cluster"])
    bad = np.argwhere(c != expect_bits(ref, "f32"))
    assert bad.size == 0, bad[:3]


@pytest.mark.parametrize("variant,shape", CASES, ids=IDS)
@pytest.mark.parametrize("ti,to", [("f16", "f32"), ("bf16", "bf16")])
def test_random_inputs_parity(variant, shape, ti, to):
    M, N, K = shape
    a, b = inputs.make_operands(M, N, K, ti, ("uniform",), ("normal", 1.0), seed=M + N + K)
    ref, S = oracle.gemm(a, b)
    c = run_variant(a, b, to, variant)
    r = parity.check(c, ref, S, to)
    assert r["ok"], r
    assert r["max_excess_rel"] < 2.0 ** -12, r   # far inside the bound: no dropped K block


@pytest.mark.parametrize("variant", [gemm.S6, gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("sched", [gemm.SCHED_STATIC, gemm.SCHED_ATOMIC, gemm.SCHED_CLC, gemm.SCHED_STREAM_K])
def test_schedulers_visit_every_tile_once(variant, sched):
    if variant == gemm.S6 and sched == gemm.SCHED_STREAM_K:
        pytest.skip("stream-K exists for the warp-specialised kernels only")
    # tile counts below, near and above the number of SMs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for M, N in [(512, 512), (2048, 2560), (4096, 4096)]:
        K = 64
        a, b = inputs.integer_operands(M, N, K, "bf16", seed=1)
        code = gemm.dtype_code("bf16", "bf16")
        plan = gemm.Plan(M, N, K, code, gemm.make_opts(variant=variant, sched=sched))
        info = plan.info()
        visits = torch.zeros(info["tiles"], dtype=torch.int32, device=DEV)
        plan.set_visits(visits)
        c = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
        for _ in range(2):   # twice: the atomic counter must rewind itself
            visits.zero_()
            plan.run(a.to(DEV), b.to(DEV), c)
            assert plan.check() == gemm.OK
            v = visits.cpu()
            assert int(v.min()) == 1 and int(v.max()) == 1, (info, sms, v.unique(return_counts=True))
        ref, _ = oracle.gemm_rows(a, b, [0, M // 2, M - 1])
        got = c.float().cpu().numpy()[[0, M // 2, M - 1]]
        assert np.array_equal(got, expect_bits(ref, "bf16"))
        plan.destroy()


@pytest.mark.parametrize("variant", [gemm.S4, gemm.S5, gemm.S7, gemm.S8, gemm.S9])
def test_forced_wait_timeout_is_reported(variant):
    M, N, K = 256, 512, 256
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=2)
    code = gemm.dtype_code("bf16", "bf16")
    plan = gemm.Plan(M, N, K, code, gemm.make_opts(variant=variant, timeout_ns=20_000_000,
                                                   debug_flags=gemm.DEBUG_SKIP_ONE_LOAD))
    c = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.ERR_DEVICE_TIMEOUT
    plan.destroy()
    # the context is still usable and the same shape computes correctly
    ref, _ = oracle.gemm(a, b)
    got = run_variant(a, b, "bf16", variant)
    assert np.array_equal(got, expect_bits(ref, "bf16"))


def test_zero_rows_give_exact_zeros():
    a, b = inputs.make_operands(300, 264, 200, "bf16", ("uniform",), ("uniform",), seed=3)
    a[5].zero_()
    a[299].zero_()
    for v in (gemm.S3, gemm.S6, gemm.S8, gemm.S9):
        c = run_variant(a, b, "bf16", v)
        assert np.all(c[5] == 0) and np.all(c[299] == 0)


def test_misaligned_pointer_rejected():
    a = torch.zeros(64 * 64 + 8, dtype=torch.bfloat16, device=DEV)
    b = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    c = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    st = gemm.gemm_run(64, 64, 64, a.data_ptr() + 2, b.data_ptr(), c.data_ptr(), gemm.BF16_BF16,
                       torch.cuda.current_stream().cuda_stream)
    assert st == gemm.ERR_MISALIGNED


def test_matmul_on_side_stream_and_auto_choices():
    a, b = inputs.make_operands(520, 776, 264, "bf16", ("uniform",), ("uniform",), seed=4)
    ref, S = oracle.gemm(a, b)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = gemm.matmul(a.to(DEV), b.to(DEV), torch.bfloat16)
    s.synchronize()
    assert parity.check(c.float().cpu().numpy(), ref, S, "bf16")["ok"]
    # odd N (rows of C not 16-byte aligned): the automatic plan still works
    a2, b2 = inputs.make_operands(200, 100, 64, "f16", ("uniform",), ("uniform",), seed=5)
    ref2, S2 = oracle.gemm(a2, b2)
    c2 = gemm.matmul(a2.to(DEV), b2.to(DEV), torch.float32)
    torch.cuda.synchronize()
    assert parity.check(c2.cpu().numpy(), ref2, S2, "f32")["ok"]
    assert gemm.gemm_check() == gemm.OK


def test_run_host_end_to_end():
    M, N, K = 300, 264, 136
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("uniform",), seed=6)
    ref, S = oracle.gemm(a, b)
    ah, bh = a.pin_memory(), b.pin_memory()
    ch = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    da = torch.empty_like(a, device=DEV)
    db = torch.empty_like(b, device=DEV)
    dc = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    st = gemm.gemm_run_host(M, N, K, ah.data_ptr(), bh.data_ptr(), ch.data_ptr(), gemm.BF16_BF16,
                            da.data_ptr(), db.data_ptr(), dc.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == gemm.OK
    assert parity.check(ch.float().numpy(), ref, S, "bf16")["ok"]


@pytest.mark.parametrize("variant,M,K", [(gemm.GEMV, 1, 512), (gemm.GEMV, 1, 1024), (gemm.GEMV, 8, 1024),
                                         (gemm.GEMV, 5, 520), (gemm.GEMV_TC, 8, 512)])
def test_static_b_flag_chains_dependent_gemvs(variant, M, K):
    """With GEMM_FLAG_STATIC_B the GEMV launches as a programmatic dependent of
    the previous kernel and may stream B early, but must read its activations
    only after that kernel is done: chain y1 = x B1^T, y2 = y1 B2^T."""
    N1 = 1024
    x, b1 = inputs.make_operands(M, N1, K, "bf16", ("uniform",), ("normal", 0.05), seed=21)
    _, b2 = inputs.make_operands(M, 768, N1, "bf16", ("uniform",), ("normal", 0.05), seed=22)
    opts = gemm.make_opts(variant=variant, flags=gemm.FLAG_STATIC_B)
    p1 = gemm.Plan(M, N1, K, gemm.BF16_BF16, opts)
    p2 = gemm.Plan(M, 768, N1, gemm.BF16_BF16, opts)
    dx, db1, db2 = x.to(DEV), b1.to(DEV), b2.to(DEV)
    y1 = torch.empty((M, N1), device=DEV, dtype=torch.bfloat16)
    y2 = torch.empty((M, 768), device=DEV, dtype=torch.bfloat16)
    for _ in range(3):
        y1.fill_(float("nan"))
        y2.fill_(float("nan"))
        p1.run(dx, db1, y1)
        p2.run(y1, db2, y2)
    torch.cuda.synchronize()
    assert p1.check() == gemm.OK and p2.check() == gemm.OK
    ref1, S1 = oracle.gemm(x, b1)
    assert parity.check(y1.float().cpu().numpy(), ref1, S1, "bf16")["ok"]
    y1h = y1.cpu()
    ref2, S2 = oracle.gemm(y1h, b2)
    assert parity.check(y2.float().cpu().numpy(), ref2, S2, "bf16")["ok"]
    p1.destroy()
    p2.destroy()


@pytest.mark.parametrize("M", [1, 8])
def test_default_gemv_reads_weights_the_previous_kernel_wrote(M):
    """Without GEMM_FLAG_STATIC_B the GEMV may ask L2 to prefetch its weights
    before the previous kernel on the stream has completed, but every value it
    uses must be the one that kernel wrote: a GEMM writes W = P Q^T, and the
    GEMV y = x W^T reads W at once.  P alternates between two integer matrices
    (W is then exact in bf16 and known from the oracle), so a stale W would
    give the other iteration's product."""
    N2, K2, KP = 1024, 2048, 16
    x, _ = inputs.make_operands(M, 8, K2, "bf16", ("uniform",), ("uniform",), seed=31)
    p_a, q = inputs.integer_operands(N2, K2, KP, "bf16", seed=32)
    p_b, _ = inputs.integer_operands(N2, K2, KP, "bf16", seed=33)
    w_ref = [torch.from_numpy(oracle.gemm(pp, q)[0]).to(torch.bfloat16) for pp in (p_a, p_b)]  # |w| <= 64: exact
    make_w = gemm.Plan(N2, K2, KP, gemm.BF16_BF16)
    gemv = gemm.Plan(M, N2, K2, gemm.BF16_BF16, gemm.make_opts(variant=gemm.GEMV))
    dx, dq = x.to(DEV), q.to(DEV)
    dps = [p_a.to(DEV), p_b.to(DEV)]
    ws = [torch.empty((N2, K2), device=DEV, dtype=torch.bfloat16) for _ in range(2)]
    ys = [torch.empty((M, N2), device=DEV, dtype=torch.bfloat16) for _ in range(4)]
    for i, y in enumerate(ys):
        w = ws[i % 2]
        w.fill_(float("nan"))
        make_w.run(dps[i % 2], dq, w)
        gemv.run(dx, w, y)
    torch.cuda.synchronize()
    assert make_w.check() == gemm.OK and gemv.check() == gemm.OK
    for k in range(2):
        assert torch.equal(ws[k].cpu(), w_ref[k])
    for i, y in enumerate(ys):
        ref, S = oracle.gemm(x, w_ref[i % 2])
        r = parity.check(y.float().cpu().numpy(), ref, S, "bf16")
        assert r["ok"], (i, r)
    make_w.destroy()
    gemv.destroy()


@pytest.mark.parametrize("M,N,K,cluster,grid", [(8, 4096, 4096, 2, 512), (5, 4104, 4096, 2, 514),
                                                 (8, 14336, 4096, 1, 1792), (3, 10000, 1032, 1, 1250)])
def test_gemv_mma_row_split_by_wave(M, N, K, cluster, grid):
    """The CUDA-core GEMV for 3 <= M <= 8 gives a cluster of two CTAs 16 weight
    rows and half of K each when those clusters fit one wave, and one CTA 8 rows
    otherwise; both forms are bit-exact on integer operands, ragged rows
    included (N % 16 == 8 for the second case)."""
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=M + N + K)
    plan = gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(variant=gemm.GEMV))
    info = plan.info()
    if info["num_sms"] == 152:
        assert (info["cluster"], info["grid"]) == (cluster, grid), info
    c = torch.empty((M, N), device=DEV)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    ref, _ = oracle.gemm(a, b)
    assert np.array_equal(c.double().cpu().numpy(), ref)
    plan.destroy()


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("stages", [2, 4, 8])
def test_gemv_tc_split_and_ring_depth(split, stages):
    M, N, K = 5, 392, 1032
    a, b = inputs.make_operands(M, N, K, "f16", ("uniform",), ("normal", 1.0), seed=split * 10 + stages)
    code = gemm.dtype_code("f16", "f32")
    plan = gemm.Plan(M, N, K, code, gemm.make_opts(variant=gemm.GEMV_TC, split_k=split, stages=stages))
    c = torch.full((M, N), float("nan"), device=DEV, dtype=torch.float32)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    assert plan.info()["cluster"] == split
    ref, S = oracle.gemm(a, b)
    r = parity.check(c.cpu().numpy(), ref, S, "f32")
    assert r["ok"], r
    plan.destroy()


def test_plans_sharing_a_kernel_keep_their_shared_memory():
    """The dynamic shared-memory limit belongs to the kernel, not the plan: a later
    plan that needs less (a shallower ring, fewer rows per CTA) must not make an
    earlier plan of the same kernel unlaunchable."""
    cases = [((512, 512, 256), gemm.make_opts(variant=gemm.S9, stages=4), gemm.make_opts(variant=gemm.S9, stages=2)),
             ((1, 1024, 512), gemm.make_opts(variant=gemm.GEMV), None)]
    for (M, N, K), o_big, o_small in cases:
        a, b = inputs.integer_operands(M, N, K, "bf16", seed=5)
        big = gemm.Plan(M, N, K, gemm.BF16_F32, o_big)
        if o_small is not None:
            small = gemm.Plan(M, N, K, gemm.BF16_F32, o_small)
            a2, b2 = a, b
        else:   # same GEMV kernel, fewer rows per CTA
            a2, b2 = inputs.integer_operands(M, 768, K, "bf16", seed=6)
            small = gemm.Plan(M, 768, K, gemm.BF16_F32, o_big)
        c1 = torch.empty((M, N), device=DEV)
        c2 = torch.empty((a2.shape[0], b2.shape[0]), device=DEV)
        for _ in range(2):
            big.run(a.to(DEV), b.to(DEV), c1)
            small.run(a2.to(DEV), b2.to(DEV), c2)
        assert big.check() == gemm.OK and small.check() == gemm.OK
        assert np.array_equal(c1.double().cpu().numpy(), oracle.gemm(a, b)[0])
        assert np.array_equal(c2.double().cpu().numpy(), oracle.gemm(a2, b2)[0])
        big.destroy()
        small.destroy()


# stream-K: shapes whose tiles outnumber the resident clusters, with several K
# blocks per tile, so that tiles are split between two clusters
SK_SHAPES = {gemm.S7: (1280, 4352, 520), gemm.S8: (1280, 4352, 264), gemm.S9: (2560, 4352, 136)}


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_stream_k_integer_bit_exact(variant, ti, to):
    M, N, K = SK_SHAPES[variant]
    a, b = inputs.integer_operands(M, N, K, ti, seed=variant)
    plan = gemm.Plan(M, N, K, gemm.dtype_code(ti, to), gemm.make_opts(variant=variant, sched=gemm.SCHED_STREAM_K))
    info = plan.info()
    assert info["sched"] == gemm.SCHED_STREAM_K and info["tiles"] > info["grid"] // info["cluster"]
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    for _ in range(3):   # repeated launches: the flags must be cleared by their consumers
        c.fill_(float("nan"))
        plan.run(a.to(DEV), b.to(DEV), c)
        assert plan.check() == gemm.OK
    plan.destroy()
    ref, _ = oracle.gemm(a, b)
    exp = expect_bits(ref, to)
    got = c.cpu().numpy() if to == "f32" else c.float().cpu().numpy()
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (info, bad[:3])


@pytest.mark.parametrize("variant", [gemm.S8, gemm.S9])
def test_stream_k_random_parity(variant):
    M, N, K = SK_SHAPES[variant]
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 1.0), seed=11 + variant)
    plan = gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(variant=variant, sched=gemm.SCHED_STREAM_K))
    c = torch.empty((M, N), device=DEV)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    ref, S = oracle.gemm(a, b)
    r = parity.check(c.cpu().numpy(), ref, S, "f32")
    assert r["ok"] and r["max_excess_rel"] < 2.0 ** -12, r


@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_automatic_stream_k_on_pairs_integer_bit_exact(ti, to):
    # a ragged few-wave output (8 x 20 pair tiles, the last row and column partial;
    # 33 K blocks, the last one partial) that the automatic plan gives step 8's
    # pairs with stream-K on 152 SMs
    M, N, K = 2000, 5000, 2056
    a, b = inputs.integer_operands(M, N, K, ti, seed=K)
    plan = gemm.Plan(M, N, K, gemm.dtype_code(ti, to))
    info = plan.info()
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert info["variant"] == gemm.S8 and info["sched"] == gemm.SCHED_STREAM_K, info
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    for _ in range(2):
        c.fill_(float("nan"))
        plan.run(a.to(DEV), b.to(DEV), c)
        assert plan.check() == gemm.OK
    plan.destroy()
    exp = expect_bits(oracle.gemm(a, b)[0], to)
    got = c.cpu().numpy() if to == "f32" else c.float().cpu().numpy()
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (info, bad[:3])


def test_stream_k_is_the_default_when_the_last_wave_is_short():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = sms // 2
    # step 9 tiles are 512 x 256: a few more tiles than CTA pairs leaves the second wave nearly empty
    p = gemm.Plan(512 * 8, 256 * ((pairs + 8) // 8), 8192, gemm.BF16_BF16)
    info = p.info()
    p.destroy()
    assert info["variant"] == gemm.S9 and info["sched"] == gemm.SCHED_STREAM_K, info
    # step 8's 256 x 256 tiles on the same output: 160 tiles fill 70 % of three waves
    p = gemm.Plan(512 * 8, 256 * ((pairs + 8) // 8), 4096, gemm.BF16_BF16)
    info = p.info()
    p.destroy()
    assert info["variant"] == gemm.S8 and info["sched"] == gemm.SCHED_STREAM_K, info
    # below 32 K blocks the partial sums cost more than the idle clusters: whole tiles
    for K in (512, 1024):
        p = gemm.Plan(512 * 8, 256 * ((pairs + 8) // 8), K, gemm.BF16_BF16)
        info = p.info()
        p.destroy()
        assert info["sched"] != gemm.SCHED_STREAM_K, info
    p = gemm.Plan(8192, 8192, 8192, gemm.BF16_BF16)
    assert p.info()["sched"] == gemm.SCHED_STATIC       # 512 tiles on 76 pairs: 96 % of seven waves
    p.destroy()


# step 9 with 224-column tiles: chosen when they finish the waves of CTA pairs sooner;
# N = 18 * 224 + 200 puts the edge inside the last 32-column band of the last tile.
# N = 4096 and 4080 (multiples of 16, 13-14 sixteen-column units per tile column) run
# 224- and 208-column tiles: 9 wide columns and 10 narrow, 8 and 11; M = 4000 leaves
# the last row of tiles ragged; M = 8192 makes four waves, each pair running four
# tiles of both widths
NARROW = [(4096, 4232, 200), (4096, 4096, 136), (4000, 4080, 200), (8192, 4080, 72)]
NARROW_TWO_WIDTHS = {4096: 9, 4080: 8}


@pytest.mark.parametrize("shape", NARROW)
@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_narrow_tiles_integer_bit_exact(shape, ti, to):
    M, N, K = shape
    a, b = inputs.integer_operands(M, N, K, ti, seed=N)
    plan = gemm.Plan(M, N, K, gemm.dtype_code(ti, to), gemm.make_opts(variant=gemm.S9))
    info = plan.info()
    assert info["variant"] == gemm.S9 and info["tile_n"] == 224, info
    if N in NARROW_TWO_WIDTHS:
        assert info["narrow_tile_n"] == 208 and info["wide_cols"] == NARROW_TWO_WIDTHS[N], info
    else:
        assert info["narrow_tile_n"] == 0, info
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    ref, _ = oracle.gemm(a, b)
    exp = expect_bits(ref, to)
    got = c.float().cpu().numpy()
    bad = np.argwhere(got != exp)
    assert bad.size == 0, (info, bad[:3])
    # the fused epilogue on the same plan runs its own 256-column tiles
    bias = torch.randint(-4, 5, (N,), generator=torch.Generator().manual_seed(1)).float()
    c2 = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    plan.run_epilogue(a.to(DEV), b.to(DEV), c2, bias=bias.to(DEV), act=gemm.ACT_RELU)
    assert plan.check() == gemm.OK
    exp2 = expect_bits(oracle.epilogue(ref, bias, None, oracle.ACT_RELU), to)
    assert np.array_equal(c2.float().cpu().numpy(), exp2)
    plan.destroy()


def test_narrow_tiles_fp8():
    M, N, K = 4096, 4232, 256
    a, b = inputs.integer_operands(M, N, K, "e4m3", seed=3, lo=-4, hi=4)
    plan = gemm.Plan(M, N, K, gemm.E4M3_BF16, gemm.make_opts(variant=gemm.S9))
    assert plan.info()["tile_n"] == 224
    c = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    ref, _ = oracle.gemm(a, b)
    assert np.array_equal(c.float().cpu().numpy(), expect_bits(ref, "bf16"))


# (4096, 4096, 4096): 8 row panels; (4096, 4104, 1024) f32: 2 panels and B split in
# halves of 2304 and 1800 columns (C is the larger transfer); (4100, 2056, 4096): ragged panels
@pytest.mark.parametrize("shape,dt", [((4096, 4096, 4096), ("bf16", "bf16")), ((4096, 4104, 1024), ("f16", "f32")),
                                      ((4100, 2056, 4096), ("bf16", "f32"))])
def test_host_entry_point_pipelines_row_panels(shape, dt):
    """gemm_run_host splits large problems into row panels whose copies overlap
    the GEMMs; every panel (and the ragged last one) must be right."""
    M, N, K = shape
    ti, to = dt
    a, b = inputs.integer_operands(M, N, K, ti, seed=M + N)
    ah, bh = a.pin_memory(), b.pin_memory()
    ch = torch.full((M, N), float("nan"), dtype=inputs.torch_dtype(to)).pin_memory()
    da, db = torch.empty_like(a, device=DEV), torch.empty_like(b, device=DEV)
    dc = torch.empty((M, N), device=DEV, dtype=inputs.torch_dtype(to))
    for _ in range(2):
        st = gemm.gemm_run_host(M, N, K, ah.data_ptr(), bh.data_ptr(), ch.data_ptr(), gemm.dtype_code(ti, to),
                                da.data_ptr(), db.data_ptr(), dc.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == gemm.OK, gemm.status_string(st)
    rows = sorted({0, 127, 128, M // 4 - 1, M // 4, M // 2, 3 * M // 4, M - 129, M - 1})
    ref, _ = oracle.gemm_rows(a, b, rows)
    got = ch[rows].double().numpy()
    assert np.array_equal(got, expect_bits(ref, to))
    assert bool(torch.isfinite(ch).all())


# stream-K with fewer tiles than clusters: every tile split between several
# consecutive clusters (the owner adds all their partials)
SMALL_OUT = [(1024, 1024, 4096, gemm.S7), (512, 4104, 4104, gemm.S7), (1024, 1024, 4096, gemm.S8),
             (1032, 1024, 2056, gemm.S9)]


@pytest.mark.parametrize("M,N,K,variant", SMALL_OUT)
@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_stream_k_small_outputs_bit_exact(M, N, K, variant, ti, to):
    a, b = inputs.integer_operands(M, N, K, ti, seed=M + K + variant)
    plan = gemm.Plan(M, N, K, gemm.dtype_code(ti, to), gemm.make_opts(variant=variant, sched=gemm.SCHED_STREAM_K))
    info = plan.info()
    assert info["sched"] == gemm.SCHED_STREAM_K and info["grid"] // info["cluster"] > info["tiles"], info
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    for _ in range(3):
        c.fill_(float("nan"))
        plan.run(a.to(DEV), b.to(DEV), c)
        assert plan.check() == gemm.OK
    plan.destroy()
    ref, _ = oracle.gemm(a, b)
    bad = np.argwhere(c.float().cpu().numpy() != expect_bits(ref, to))
    assert bad.size == 0, (info, bad[:3])


def test_stream_k_small_output_random_parity():
    M, N, K = 768, 2048, 8192
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 1.0), seed=5)
    plan = gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(sched=gemm.SCHED_STREAM_K))
    assert plan.info()["sched"] == gemm.SCHED_STREAM_K
    c = torch.empty((M, N), device=DEV)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    ref, S = oracle.gemm(a, b)
    r = parity.check(c.cpu().numpy(), ref, S, "f32")
    assert r["ok"] and r["max_excess_rel"] < 2.0 ** -12, r


# step 7 with K split over a cluster (partials exchanged over distributed shared memory for two
# CTAs, through the plan's L2-resident workspace for more)
KS_CASES = [(1024, 1024, 4096, 0), (512, 1024, 8192, 0), (256, 512, 2048, 0), (300, 520, 1040, 2),
            (129, 1288, 2056, 3), (640, 264, 4104, 5), (256, 512, 8192, 8)]
# automatic split: as many slices per tile as the SMs hold (152 SMs) with every cluster
# resident at once, at most 4, each keeping >= 16 K blocks; the automatic plan takes step 8's
# CTA pairs unless they would occupy fewer SMs (1024 x 1024 x 4096 stays on step 7)
KS_AUTO = {(1024, 1024, 4096): 4, (512, 1024, 8192): 4, (256, 512, 2048): 2}


# step 8's 256 x 256 tile on a CTA pair with K split into 2-4 slices (clusters of 4-8 CTAs)
KS_PAIR_CASES = [(1024, 1024, 4096, 4), (512, 4096, 4096, 2), (300, 520, 1040, 2), (129, 1288, 2056, 3),
                 (640, 264, 4104, 4), (256, 512, 8192, 4)]
KS_AUTO_PAIR = {(1024, 1024, 4096): 3, (512, 1024, 8192): 4, (256, 512, 2048): 2}


@pytest.mark.parametrize("M,N,K,split,variant", [c + (gemm.S7,) for c in KS_CASES] +
                         [c + (gemm.S8,) for c in KS_PAIR_CASES])
@pytest.mark.parametrize("ti,to", [("bf16", "bf16"), ("f16", "f32")])
def test_split_k_cluster_bit_exact(M, N, K, split, variant, ti, to):
    a, b = inputs.integer_operands(M, N, K, ti, seed=M + split)
    plan = gemm.Plan(M, N, K, gemm.dtype_code(ti, to), gemm.make_opts(variant=variant if split else 0, split_k=split))
    info = plan.info()
    if split:
        assert info["variant"] == variant, info
    cg = 2 if info["variant"] == gemm.S8 else 1
    auto = KS_AUTO_PAIR if cg == 2 else KS_AUTO
    assert info["variant"] in (gemm.S7, gemm.S8) and info["cluster"] == cg * (split or auto[(M, N, K)]), info
    assert info["grid"] == info["tiles"] * info["cluster"], info
    visits = torch.zeros(info["tiles"], dtype=torch.int32, device=DEV)
    plan.set_visits(visits)
    c = torch.full((M, N), float("nan"), device=DEV, dtype=inputs.torch_dtype(to))
    for _ in range(2):
        visits.zero_()
        c.fill_(float("nan"))
        plan.run(a.to(DEV), b.to(DEV), c)
        assert plan.check() == gemm.OK
        assert int(visits.min()) == 1 and int(visits.max()) == 1
    plan.destroy()
    ref, _ = oracle.gemm(a, b)
    bad = np.argwhere(c.float().cpu().numpy() != expect_bits(ref, to))
    assert bad.size == 0, (info, bad[:3])


def test_split_k_cluster_random_parity_and_refusals():
    M, N, K = 512, 4096, 4096
    a, b = inputs.make_operands(M, N, K, "bf16", ("uniform",), ("normal", 1.0), seed=9)
    plan = gemm.Plan(M, N, K, gemm.BF16_F32)
    info = plan.info()
    assert (info["variant"], info["cluster"]) in ((gemm.S7, 2), (gemm.S8, 4)), info
    c = torch.empty((M, N), device=DEV)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    ref, S = oracle.gemm(a, b)
    r = parity.check(c.cpu().numpy(), ref, S, "f32")
    assert r["ok"] and r["max_excess_rel"] < 2.0 ** -12, r
    with pytest.raises(gemm.GemmError):
        gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(variant=gemm.S9, split_k=2))
    p1 = gemm.Plan(M, N, K, gemm.BF16_F32, gemm.make_opts(split_k=1))
    i1 = p1.info()
    assert i1["cluster"] == (2 if i1["variant"] == gemm.S8 else 1), i1  # no K split
    p1.destroy()
    # a forced split whose workspace (128 KB per CTA) would exceed 512 MB:
    # 64 x 32 tiles x 8 CTAs
    with pytest.raises(gemm.GemmError):
        gemm.Plan(8192, 8192, 1024, gemm.BF16_BF16, gemm.make_opts(variant=gemm.S7, split_k=8))


# extreme aspect ratios: a 65536-deep K loop, 512 tile columns of one tile row, 256 tile rows
# of one (ragged) tile column; integer operands make every result exact
EXTREME = [(256, 256, 65536), (128, 131072, 64), (131072, 136, 64)]


@pytest.mark.parametrize("M,N,K", EXTREME)
def test_extreme_shapes_bit_exact(M, N, K):
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=K + 1)
    info = []
    c = run_variant(a, b, "bf16", 0, plan_out=info)
    ref, _ = oracle.gemm(a, b)
    bad = np.argwhere(c != expect_bits(ref, "bf16"))
    assert bad.size == 0, (info, bad[:3])


def test_output_of_more_than_2_31_elements():
    # C is 65536 x 65536 bf16 (8 GiB): row offsets past 2^31 elements need 64-bit
    # addressing in every store path; sampled rows against the oracle, all of C finite
    M = N = 65536
    K = 64
    a, b = inputs.integer_operands(M, N, K, "bf16", seed=3)
    plan = gemm.Plan(M, N, K, gemm.BF16_BF16)
    c = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
    plan.run(a.to(DEV), b.to(DEV), c)
    assert plan.check() == gemm.OK
    plan.destroy()
    assert bool(torch.isfinite(c).all())
    rows = [0, 1, 32767, 32768, 40000, 65534, 65535]
    ref, _ = oracle.gemm_rows(a, b, rows)
    got = c[rows].float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, expect_bits(ref, "bf16"))
    del c
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", [gemm.S7, gemm.S8, gemm.S9])
def test_back_to_back_dependent_gemms(variant):
    # Steps 7-9 launch as programmatic dependents of the previous kernel. Each GEMM
    # here reads the one before it (as A, and as the residual of a fused epilogue),
    # and the last one overwrites a buffer the third reads, all on one stream with
    # no host synchronisation: every launch must see the finished data and must not
    # overwrite what its predecessor still reads. Integer operands keep every fp32
    # sum exact, so each bf16 result is unique.
    M, K1, N1, N2 = 2048, 64, 256, 64
    a, b1 = inputs.integer_operands(M, N1, K1, "bf16", seed=1)
    _, b2 = inputs.integer_operands(8, N2, N1, "bf16", seed=2)
    _, b3 = inputs.integer_operands(8, N1, N2, "bf16", seed=3, lo=-1, hi=1)
    _, b4 = inputs.integer_operands(8, N1, K1, "bf16", seed=4)
    opts = gemm.make_opts(variant=variant)
    p1, p2, p3 = (gemm.Plan(M, n, k, gemm.BF16_BF16, opts) for n, k in ((N1, K1), (N2, N1), (N1, N2)))
    da, d1, d2, d3, d4 = (x.to(DEV) for x in (a, b1, b2, b3, b4))
    c1 = torch.empty((M, N1), device=DEV, dtype=torch.bfloat16)
    c2 = torch.empty((M, N2), device=DEV, dtype=torch.bfloat16)
    c3 = torch.empty((M, N1), device=DEV, dtype=torch.bfloat16)
    for _ in range(3):
        c1.fill_(float("nan")), c2.fill_(float("nan")), c3.fill_(float("nan"))
        torch.cuda.synchronize()
        p1.run(da, d1, c1)                        # c1 = a b1^T
        p2.run(c1, d2, c2)                        # c2 = c1 b2^T
        p3.run_epilogue(c2, d3, c3, residual=c1)  # c3 = c2 b3^T + c1
        p1.run(da, d4, c1)                        # c1 = a b4^T, after c1 was read
        torch.cuda.synchronize()
        for p in (p1, p2, p3):
            assert p.check() == gemm.OK
        r1 = expect_bits(oracle.gemm(a, b1)[0], "bf16")
        r2 = expect_bits(oracle.gemm(torch.tensor(r1).to(torch.bfloat16), b2)[0], "bf16")
        pre3, _ = oracle.gemm(torch.tensor(r2).to(torch.bfloat16), b3)
        r3 = expect_bits(pre3 + r1, "bf16")
        r4 = expect_bits(oracle.gemm(a, b4)[0], "bf16")
        assert np.array_equal(c2.float().cpu().numpy(), r2)
        assert np.array_equal(c3.float().cpu().numpy(), r3)
        assert np.array_equal(c1.float().cpu().numpy(), r4)
    for p in (p1, p2, p3):
        p.destroy()


def test_dependent_gemms_captured_in_a_cuda_graph():
    # the programmatic launch of steps 7-9 inside stream capture: two GEMMs, the
    # second reading the first's output, captured once and replayed
    M, K1, N1, N2 = 2048, 64, 512, 64
    a, b1 = inputs.integer_operands(M, N1, K1, "bf16", seed=21)
    _, b2 = inputs.integer_operands(8, N2, N1, "bf16", seed=22)
    opts = gemm.make_opts(variant=gemm.S9)
    p1, p2 = gemm.Plan(M, N1, K1, gemm.BF16_BF16, opts), gemm.Plan(M, N2, N1, gemm.BF16_BF16, opts)
    da, d1, d2 = a.to(DEV), b1.to(DEV), b2.to(DEV)
    c1 = torch.empty((M, N1), device=DEV, dtype=torch.bfloat16)
    c2 = torch.empty((M, N2), device=DEV, dtype=torch.bfloat16)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p1.run(da, d1, c1, stream=s)   # first use outside the capture (operand descriptors)
        p2.run(c1, d2, c2, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        p1.run(da, d1, c1, stream=s)
        p2.run(c1, d2, c2, stream=s)
    r1 = expect_bits(oracle.gemm(a, b1)[0], "bf16")
    r2 = expect_bits(oracle.gemm(torch.tensor(r1).to(torch.bfloat16), b2)[0], "bf16")
    for _ in range(3):
        c1.fill_(float("nan"))
        c2.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert p1.check() == gemm.OK and p2.check() == gemm.OK
        assert np.array_equal(c1.float().cpu().numpy(), r1)
        assert np.array_equal(c2.float().cpu().numpy(), r2)
    del g
    p1.destroy()
    p2.destroy()
