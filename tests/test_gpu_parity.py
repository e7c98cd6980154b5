"""Parity of the sm_103a GEMM (through the C ABI) with the CPU oracle.

Every case compares the GPU result element by element with the oracle on the
same seeded fp16 inputs, under |C_gpu - C_ref| <= 2 ulp16(|C_ref|) + 1e-4 sqrt(K)
(bit-exact for small-integer inputs).  C is pre-filled with NaN so an element
the kernel fails to write shows up, and padding columns/rows of every buffer
must come back untouched.  After each case the device watchdog word must be 0.
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, lib_for, to_device, to_host
from tests.tolerance import check_bitexact, check_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"
    if "mcast" in g._libs:   # the multicast build has a watchdog word of its own
        assert g.device_status(lib=g.library_mcast()) == 0, "watchdog word set after the case"


def run(A, B, *, lda=None, ldb=None, ldc=None, extra_rows=0, options=None, stream=None):
    M, K = A.shape
    N, _ = B.shape
    Ad = to_device(A, lda)
    Bd = to_device(B, ldb)
    Cd, Cbuf = empty_out(M, N, ldc, extra_rows)
    g.gemm_f16_nt(Ad, Bd, Cd, options=options, stream=stream,
                  lib=lib_for(options.cluster_pairs if options is not None else 0))
    torch.cuda.synchronize()
    # margins: padding columns and extra rows of C untouched (still NaN)
    pad = to_host(Cbuf)
    assert np.isnan(pad[:M, N:].astype(np.float32)).all(), "padding columns of C were written"
    assert np.isnan(pad[M:, :].astype(np.float32)).all(), "rows past M were written"
    return to_host(Cd)


def opts(cg, **kw):
    return g.Options(cta_group=cg, **kw)


SMALL = [(128, 256, 64), (256, 256, 256), (1, 1, 1), (1, 1, 8), (7, 9, 3), (300, 520, 328),
         (513, 1025, 200), (1000, 700, 1000), (129, 257, 65), (64, 8, 4096), (255, 511, 63),
         (2, 1000, 130)]


@pytest.mark.parametrize("cg", [2, 1])
@pytest.mark.parametrize("M,N,K", SMALL)
def test_small_shapes(M, N, K, cg):
    A = inputs.draw((M, K), inputs.U, 11 + M)
    B = inputs.draw((N, K), inputs.U, 13 + N)
    C = run(A, B, options=opts(cg))
    check_close(C, oracle.gemm_f16_nt(A, B), K, f"{M}x{N}x{K} cg{cg}")


@pytest.mark.parametrize("cg,max_clusters,swizzle", [(2, 1, 1), (2, 3, 3), (2, 5, 8), (2, 7, 64),
                                                     (1, 1, 2), (1, 5, 8), (1, 11, 1)])
def test_persistent_loop_many_tiles_per_cta(cg, max_clusters, swizzle):
    # every CTA walks many tiles: ring phases and both TMEM buffers wrap many times
    M, N, K = 1100, 2100, 520
    A = inputs.draw((M, K), inputs.U, 21)
    B = inputs.draw((N, K), inputs.U, 22)
    C = run(A, B, options=opts(cg, max_clusters=max_clusters, swizzle=swizzle))
    check_close(C, oracle.gemm_f16_nt(A, B), K, f"persistent cg{cg} mc{max_clusters} sw{swizzle}")


@pytest.mark.parametrize("cg,max_clusters,shape", [
    (2, 7, (1100, 2100, 520)),     # 45 tiles on 7 pairs: 3 left over + 7 split in k
    (2, 5, (1100, 2100, 520)),     # 45 % 5 == 0: forced split of one full wave
    (2, 0, (256, 256, 4096)),      # one tile split over 64 pairs: 63 partials per owner
    (2, 0, (700, 900, 1500)),      # 12 tiles over many pairs, ragged edges
    (1, 9, (1000, 1100, 700)),     # single-CTA tiles
    (1, 0, (130, 300, 2048)),
])
def test_stream_k_split_tiles(cg, max_clusters, shape):
    M, N, K = shape
    A = inputs.draw((M, K), inputs.U, 91 + M)
    B = inputs.draw((N, K), inputs.U, 92 + N)
    o = opts(cg, max_clusters=max_clusters, schedule=2)
    pl = g.plan(M, N, K, options=o)
    assert pl["sk_tiles"] > 0
    C1 = run(A, B, options=o)
    check_close(C1, oracle.gemm_f16_nt(A, B), K, f"stream-K {shape} cg{cg}")
    C2 = run(A, B, options=o)                      # partials are summed in a fixed order
    assert np.array_equal(C1.view(np.uint16), C2.view(np.uint16))


@pytest.mark.parametrize("shape,max_clusters,schedule,split", [
    ((1100, 2100, 520), 7, 3, 2),   # forced: 45 tiles on 7 pairs, the last 3 cut in two
    ((1100, 2100, 520), 20, 3, 4),  # forced: the last 5 cut in four; N = 2100: slices past N store nothing
    ((300, 520, 328), 0, 0, 4),     # 6 tiles of 6 k-blocks, all cut in four, over 24 pairs
    ((1, 1, 1), 0, 0, 4),
    ((1536, 1000, 256), 0, 0, 2),   # 24 tiles: cut in two; N % 8 == 0, M edge exact
    ((513, 1025, 200), 9, 3, 1),    # 15 tiles on 9 pairs: 6 left over, 6·2 > 9: no split
])
def test_n_split(shape, max_clusters, schedule, split):
    M, N, K = shape
    A = inputs.draw((M, K), inputs.U, 95 + M)
    B = inputs.draw((N, K), inputs.U, 96 + N)
    # (cta_group 2: the persistent kernel; small problems default to the small-problem kernel)
    o = g.Options(cluster_pairs=1, cta_group=2, max_clusters=max_clusters, schedule=schedule)
    pl = g.plan(M, N, K, options=o)
    assert pl["tail_split"] == split and pl["sk_tiles"] == 0
    C = run(A, B, options=o)
    check_close(C, oracle.gemm_f16_nt(A, B), K, f"N-split {shape}")
    # each output's k order is the same whatever the MMA width: identical to whole tiles
    whole = run(A, B, options=g.Options(cluster_pairs=1, cta_group=2, max_clusters=max_clusters, schedule=1))
    assert np.array_equal(C.view(np.uint16), whole.view(np.uint16))


def test_n_split_integers_and_fp16_accumulator():
    M, N, K = 1300, 1000, 320                     # 24 tiles of 5 k-blocks: all cut in two
    A = inputs.draw((M, K), inputs.I2, 97)
    B = inputs.draw((N, K), inputs.I2, 98)
    one = g.Options(cluster_pairs=1, cta_group=2)
    assert g.plan(M, N, K, options=one)["tail_split"] == 2
    check_bitexact(run(A, B, options=one), oracle.gemm_f16_nt(A, B), "N-split int")
    A16 = (A * (np.arange(K) % 4 == 0)).astype(np.float16)   # partial sums exact in fp16
    C16 = run(A16, B, options=g.Options(cluster_pairs=1, accumulate=1))
    assert np.array_equal(C16.astype(np.float64), A16.astype(np.float64) @ B.astype(np.float64).T)


@pytest.mark.parametrize("shape,max_clusters,schedule", [
    ((1100, 2100, 520), 0, 0),      # 5 x 5 cluster tiles of 256 x 512
    ((1100, 2100, 520), 2, 1),      # persistent: 12-13 cluster tiles per cluster
    ((513, 1300, 200), 0, 2),       # odd number of 256-wide N tiles: pair 1 out of range
    ((256, 300, 4096), 0, 2),       # one cluster tile split in k over many clusters
    ((4000, 3000, 5000), 0, 0),     # the ragged workload shape
    ((7, 9, 3), 0, 0),
])
def test_two_pairs_per_cluster_a_multicast(shape, max_clusters, schedule):
    M, N, K = shape
    A = inputs.draw((M, K), inputs.U, 71 + M)
    B = inputs.draw((N, K), inputs.U, 72 + N)
    o = g.Options(cluster_pairs=2, max_clusters=max_clusters, schedule=schedule)
    C = run(A, B, options=o)
    check_close(C, oracle.gemm_f16_nt(A, B), K, f"two pairs {shape}")


def test_two_pairs_integers_bit_exact():
    M, N, K = 1000, 1500, 2000
    A = inputs.draw((M, K), inputs.I2, 73)
    B = inputs.draw((N, K), inputs.I2, 74)
    check_bitexact(run(A, B, options=g.Options(cluster_pairs=2)), oracle.gemm_f16_nt(A, B), "two pairs int")


def test_alternating_k_order_rounds():
    """Whole tiles of odd rounds load their k-blocks from the last one down
    (plan k_order 1): two rounds of 16 clusters at K = 16384, float inputs
    against the oracle and integer inputs bit-exact."""
    M, N, K = 1024, 2048, 16384
    o = opts(2, max_clusters=16)
    pl = g.plan(M, N, K, options=o)
    assert (pl["k_order"], pl["num_tiles"], pl["clusters"], pl["sk_tiles"], pl["tail_split"]) == (1, 32, 16, 0, 1)
    A = inputs.draw((M, K), inputs.U, 131)
    B = inputs.draw((N, K), inputs.U, 132)
    check_close(run(A, B, options=o), oracle.gemm_f16_nt(A, B), K, "alternating k order")
    Ai = inputs.draw((M, K), inputs.I2, 133)
    Bi = inputs.draw((N, K), inputs.I2, 134)
    check_bitexact(run(Ai, Bi, options=o), oracle.gemm_f16_nt(Ai, Bi), "alternating k order int")


@pytest.mark.parametrize("cg,M,N,K,mc", [(2, 1100, 2100, 520, 7), (1, 700, 900, 1000, 5), (2, 4000, 3000, 600, 20)])
def test_claimed_last_wave(cg, M, N, K, mc):
    """The tiles of a last, partial wave are claimed at run time by the clusters
    that finish first (one each at most): float inputs against the oracle,
    the same bits on every repeat whichever clusters took them, integer inputs
    bit-exact."""
    o = opts(cg, max_clusters=mc, schedule=1)
    pl = g.plan(M, N, K, options=o)
    assert pl["claimed_tiles"] == pl["num_tiles"] % pl["clusters"] > 0
    A = inputs.draw((M, K), inputs.U, 141 + M)
    B = inputs.draw((N, K), inputs.U, 142 + N)
    C1 = run(A, B, options=o)
    check_close(C1, oracle.gemm_f16_nt(A, B), K, f"claimed last wave {M}x{N}x{K} cg{cg}")
    for _ in range(4):
        assert np.array_equal(run(A, B, options=o).view(np.uint16), C1.view(np.uint16))
    Ai = inputs.draw((M, K), inputs.I2, 143 + M)
    Bi = inputs.draw((N, K), inputs.I2, 144 + N)
    check_bitexact(run(Ai, Bi, options=o), oracle.gemm_f16_nt(Ai, Bi), f"claimed last wave int cg{cg}")


def test_stream_k_integers_bit_exact_and_matches_whole_tiles():
    M, N, K = 1200, 1000, 2200
    A = inputs.draw((M, K), inputs.I2, 93)
    B = inputs.draw((N, K), inputs.I2, 94)
    ref = oracle.gemm_f16_nt(A, B)
    sk = run(A, B, options=opts(2, max_clusters=6, schedule=2))
    dp = run(A, B, options=opts(2, max_clusters=6, schedule=1))
    check_bitexact(sk, ref, "stream-K int")
    check_bitexact(dp, ref, "whole tiles int")


@pytest.mark.parametrize("cg", [2, 1])
def test_leading_dimensions_and_margins(cg):
    # N % 8 != 0: the last columns are not a whole 16-byte unit of C's rows
    M, N, K = 333, 601, 250
    A = inputs.draw((M, K), inputs.U, 31)
    B = inputs.draw((N, K), inputs.U, 32)
    C = run(A, B, lda=K + 6 + 24, ldb=K + 6 + 8, ldc=N + 47, extra_rows=5, options=opts(cg))
    check_close(C, oracle.gemm_f16_nt(A, B), K, "pitched")


@pytest.mark.parametrize("cg", [2, 1])
def test_integer_inputs_bit_exact_small(cg):
    M, N, K = 700, 900, 3000
    A = inputs.draw((M, K), inputs.I2, 41)
    B = inputs.draw((N, K), inputs.I2, 42)
    check_bitexact(run(A, B, options=opts(cg)), oracle.gemm_f16_nt(A, B), "int small")


def test_identity_and_permutation_exact():
    K = 512
    A = inputs.draw((384, K), inputs.U, 51)
    eye = np.eye(K, dtype=np.float16)
    check_bitexact(run(A, eye), A, "identity")
    pi = np.random.default_rng(3).permutation(K)
    P = np.zeros((K, K), dtype=np.float16)
    P[np.arange(K), pi] = 1.0
    check_bitexact(run(A, P), A[:, pi], "permutation")


def test_k_zero_writes_positive_zero():
    M, N = 300, 200
    Cd, Cbuf = empty_out(M, N, extra_rows=3)
    Ad = torch.empty((M, 0), dtype=torch.float16, device="cuda:0")
    Bd = torch.empty((N, 0), dtype=torch.float16, device="cuda:0")
    g.gemm_f16_nt(Ad, Bd, Cd)
    torch.cuda.synchronize()
    c = to_host(Cd)
    assert np.all(c.view(np.uint16) == 0)
    assert np.isnan(to_host(Cbuf)[M:].astype(np.float32)).all()


def test_empty_output_is_a_noop():
    Cd, _ = empty_out(0, 64)
    g.gemm_f16_nt(torch.empty((0, 64), dtype=torch.float16, device="cuda:0"),
                  torch.empty((64, 64), dtype=torch.float16, device="cuda:0"), Cd)
    torch.cuda.synchronize()


def test_misaligned_device_pointer_rejected():
    A = torch.zeros((64, 72), dtype=torch.float16, device="cuda:0")
    B = torch.zeros((64, 64), dtype=torch.float16, device="cuda:0")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(A[:, 1:65], B)          # starts 2 bytes into a row
    assert e.value.status == 2


def test_repeat_is_deterministic_and_other_stream():
    M, N, K = 1024, 768, 1536
    A = inputs.draw((M, K), inputs.U, 61)
    B = inputs.draw((N, K), inputs.U, 62)
    c1 = run(A, B)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c2 = run(A, B, stream=s)
    assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))


def test_output_error_scale_unit_variance_k8192():
    # Tilus tutorial, "6. Register Reallocation, Multicast, and a Persistent
    # Kernel", §Shared-Memory Epilogue (Note): with fp32 accumulation and
    # unit-variance outputs at K = 8192 the mean absolute error is 0.00014.
    M, N, K = 512, 512, 8192
    s = K ** -0.25
    A = inputs.draw((M, K), ("normal", 0.0, s), 71)
    B = inputs.draw((N, K), ("normal", 0.0, s), 72)
    C = run(A, B).astype(np.float64)
    S = oracle.gemm_f16_nt_f64(A, B)
    mae = np.abs(C - S).mean()
    assert 1.0e-4 < mae < 1.8e-4, mae
    check_close(C.astype(np.float16), oracle.gemm_f16_nt(A, B), K, "unit variance")


# ---------------------------------------------------------------------------
# the benchmark workloads at full size
# ---------------------------------------------------------------------------

def sample_points(M, N, n_random=3000, seed=0):
    """Corners, tile edges (multiples of 128/256 and their neighbours) and random
    positions."""
    rng = np.random.default_rng(seed)
    edge_r = sorted({0, 1, M - 1, M - 2} | {min(max(v + d, 0), M - 1)
                                               for v in range(0, M, 128) for d in (-1, 0)})
    edge_c = sorted({0, 1, N - 1, N - 2} | {min(max(v + d, 0), N - 1)
                                               for v in range(0, N, 256) for d in (-1, 0)})
    rr = rng.choice(edge_r, 400)
    cc = rng.choice(edge_c, 400)
    rows = np.concatenate([rr, rng.integers(0, M, n_random), [0, 0, M - 1, M - 1]])
    cols = np.concatenate([cc, rng.integers(0, N, n_random), [0, N - 1, 0, N - 1]])
    return rows, cols


def run_workload(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.operands(w)
    Ad, Bd = to_device(A), to_device(B)
    Cd, _ = empty_out(w.M, w.N)
    g.gemm_f16_nt(Ad, Bd, Cd)
    torch.cuda.synchronize()
    return w, A, B, Cd


@pytest.mark.parametrize("name", ["gemm_256", "gemm_4096", "ragged_4000x3000x5000", "gemm_8192",
                                  "mlp_up_16384x14336x4096"])
def test_workload_full_check(name):
    """Every element of every float workload at full size against the oracle
    (8192^3 and the MLP shape take the oracle tens of seconds on the host)."""
    w, A, B, Cd = run_workload(name)
    C = to_host(Cd)
    del Cd
    check_close(C, oracle.gemm_f16_nt(A, B), w.K, name)


def test_workload_ragged_integers_bit_exact():
    w, A, B, Cd = run_workload("ragged_int_4000x3000x5000")
    check_bitexact(to_host(Cd), oracle.gemm_f16_nt(A, B), w.name)


# ---------------------------------------------------------------------------
# maximum sizes: 64-bit offsets, a very long k loop, a very tall problem
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,why", [
    (70000, 32768, 64, "C is 4.6 GB: row offsets past 2^31 elements"),
    (256, 512, 1 << 20, "2^20-deep k loop, split in k over every pair"),
    (1 << 20, 72, 128, "a million rows, N % 64 != 0"),
])
def test_maximum_sizes_sampled(M, N, K, why):
    A = inputs.draw((M, K), inputs.U, 601 + M % 97)
    B = inputs.draw((N, K), inputs.U, 602 + N % 97)
    Ad, Bd = to_device(A), to_device(B)
    Cd, _ = empty_out(M, N)
    g.gemm_f16_nt(Ad, Bd, Cd)
    torch.cuda.synchronize()
    assert not torch.isnan(Cd).any().item(), f"unwritten (NaN) elements in C ({why})"
    rows, cols = sample_points(M, N, n_random=2000 if K < 4096 else 200)
    if K >= 4096:   # each point is a 2^20-term dot product on the host: keep the sample small
        keep = np.random.default_rng(1).choice(rows.size, 300, replace=False)
        rows, cols = rows[keep], cols[keep]
    got = Cd[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    ref, _ = oracle.gemm_f16_nt_points(A, B, rows, cols)
    check_close(got, ref, K, why)
    del Cd, Ad, Bd
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# operand layouts: A stored [K, M] and/or B stored [K, N] (MN-major tiles)
# ---------------------------------------------------------------------------

def run_layout(A_mk, B_nk, a_layout, b_layout, options, bf16=False):
    """Store A / B in the requested layout (padded pitch), run, return C."""
    M, K = A_mk.shape
    N = B_nk.shape[0]
    A_st = np.ascontiguousarray(A_mk.T) if a_layout else A_mk
    B_st = np.ascontiguousarray(B_nk.T) if b_layout else B_nk
    lda = A_st.shape[1] + 8 + (-A_st.shape[1]) % 8
    ldb = B_st.shape[1] + 16 + (-B_st.shape[1]) % 8
    Ad, Bd = to_device(A_st, lda), to_device(B_st, ldb)
    Cd, Cbuf = empty_out(M, N, extra_rows=2)
    options.a_layout, options.b_layout = a_layout, b_layout
    g.gemm_f16_nt_ptr(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), Cbuf.stride(0),
                      torch.cuda.current_stream().cuda_stream, options, lib=lib_for(options.cluster_pairs))
    torch.cuda.synchronize()
    assert np.isnan(to_host(Cbuf)[M:].astype(np.float32)).all(), "rows past M were written"
    return to_host(Cd)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("cg,cp", [(2, 1), (1, 1), (2, 2)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 328), (1000, 1100, 700)])
def test_operand_layouts(M, N, K, cg, cp, a_layout, b_layout):
    A = inputs.draw((M, K), inputs.U, 501 + M)
    B = inputs.draw((N, K), inputs.U, 502 + N)
    C = run_layout(A, B, a_layout, b_layout, g.Options(cta_group=cg, cluster_pairs=cp))
    check_close(C, oracle.gemm_f16_nt(A, B), K, f"layout A{a_layout} B{b_layout} cg{cg} cp{cp}")


def test_operand_layouts_stream_k_and_integers():
    M, N, K = 700, 900, 3000
    A = inputs.draw((M, K), inputs.I2, 503)
    B = inputs.draw((N, K), inputs.I2, 504)
    ref = oracle.gemm_f16_nt(A, B)
    for al, bl in ((0, 1), (1, 0), (1, 1)):
        check_bitexact(run_layout(A, B, al, bl, g.Options(schedule=2, max_clusters=5)), ref,
                       f"layout A{al} B{bl} stream-K int")


def test_layout_pitch_rule():
    # a [K, M] A needs lda >= M, not lda >= K
    A = torch.zeros((64, 256), dtype=torch.float16, device="cuda:0")      # K=64 rows of M=256
    B = torch.zeros((512, 64), dtype=torch.float16, device="cuda:0")
    C = torch.empty((256, 512), dtype=torch.float16, device="cuda:0")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_ptr(256, 512, 64, A.data_ptr(), 128, B.data_ptr(), 64, C.data_ptr(), 512, 0,
                          g.Options(a_layout=1))
    assert e.value.status == 1


# ---------------------------------------------------------------------------
# split pieces: every tile cut along k into s pieces that reduce each other
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shape,max_clusters,pieces", [
    ((1024, 1024, 1024), 0, 4),     # 16 tiles of 16 k-blocks over 64 pairs
    ((1024, 1024, 1024), 32, 2),    # the same over 32 pairs
    ((256, 256, 8192), 0, 8),       # one tile, 8 pieces of 16 k-blocks
    ((300, 520, 328), 0, 4),        # 6 ragged tiles of 6 k-blocks: uneven pieces (1 or 2 k-blocks)
    ((513, 1100, 2000), 0, 4),      # N % 8 != 0: the last 32-column slice stored element-wise
    ((1, 1, 100), 0, 2),            # 2 k-blocks, one valid row and column
])
def test_split_pieces(shape, max_clusters, pieces):
    M, N, K = shape
    A = inputs.draw((M, K), inputs.U, 801 + M)
    B = inputs.draw((N, K), inputs.U, 802 + N)
    o = g.Options(max_clusters=max_clusters, schedule=4)
    pl = g.plan(M, N, K, options=o)
    assert pl["split_pieces"] == pieces and pl["sk_tiles"] == 0
    C1 = run(A, B, options=o)
    check_close(C1, oracle.gemm_f16_nt(A, B), K, f"split pieces {shape}")
    C2 = run(A, B, options=o)                      # the pieces are summed in a fixed order
    assert np.array_equal(C1.view(np.uint16), C2.view(np.uint16))


@pytest.mark.parametrize("cg", [2, 1])
def test_split_pieces_integers_bit_exact(cg):
    M, N, K = 700, 900, 3000
    A = inputs.draw((M, K), inputs.I2, 803)
    B = inputs.draw((N, K), inputs.I2, 804)
    o = g.Options(cta_group=cg, schedule=4)
    assert g.plan(M, N, K, options=o)["split_pieces"] > 1
    check_bitexact(run(A, B, options=o), oracle.gemm_f16_nt(A, B), f"split pieces int cg{cg}")
