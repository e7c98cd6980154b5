"""The small-problem kernel (one 128·cta_group × tile_n tile of C per cluster,
all of k in one CTA or CTA pair) against the oracle, through the C ABI.

Forced (schedule 5) for both CTA groups and every tile width on shapes with
ragged edges in M, N and K, k deep enough for the stage ring to wrap several
times, and padded pitches whose padding holds NaN (a read of it would poison
the result); C's padding columns and a row past M must come back untouched.
Chosen by default for small problems (checked through the launch plan), also
under stream capture, where it needs no workspace; with few tiles and deep k
it splits each tile along k (split-K, owner adds the pieces in k order).  Bars as everywhere:
small-integer inputs bit-exact, others within 2 ulps of the output format +
1e-4·sqrt(K).
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, to_device, to_host
from tests.tolerance import bf16_to_f64, check_bitexact, check_close, ulp_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402

NAN16, NANBF = 0x7E00, 0x7FC0
VARIANTS = [(cg, bn) for cg in (1, 2) for bn in (32, 64, 128)]
SHAPES = [
    (300, 520, 328),     # ragged in M, N and K; several tiles each way
    (1, 8, 1),           # one row, one 8-column group, one k
    (129, 33, 65),       # one row into the second M tile, N % 8 != 0, two k-blocks
    (257, 200, 1000),    # M one past two CTA tiles, 16 k-blocks (the ring wraps)
    (256, 192, 4096),    # 64 k-blocks: the ring wraps 8 times
]
_ref_cache = {}


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def _operands(M, N, K, ints):
    dist = inputs.I2 if ints else inputs.U
    return inputs.draw((M, K), dist, 4100 + M + K), inputs.draw((N, K), dist, 4200 + N + K)


def _reference(M, N, K, ints):
    key = (M, N, K, ints)
    if key not in _ref_cache:
        A, B = _operands(M, N, K, ints)
        _ref_cache[key] = (A, B, oracle.gemm_f16_nt(A, B))
    return _ref_cache[key]


def _run(A, B, options, pad=(8, 16, 8), bf16=False):
    """A, B as 16-bit patterns (uint16) in pitched NaN-padded buffers; returns C's
    bits and checks the padding columns and the extra row past M."""
    M, K = A.shape
    N = B.shape[0]
    r8 = lambda v: v + (-v) % 8
    lda, ldb, ldc = r8(K) + pad[0], r8(K) + pad[1], r8(N) + pad[2]
    nan = NANBF if bf16 else NAN16

    def dev(bits, ld, rows):
        buf = np.full((max(rows, 1), ld), nan, dtype=np.uint16)
        buf[:bits.shape[0], :bits.shape[1]] = bits
        return torch.from_numpy(buf.view(np.int16)).cuda()

    Ad, Bd, Cd = dev(A, lda, M), dev(B, ldb, N), dev(np.zeros((0, 0), np.uint16), ldc, M + 1)
    g.gemm_f16_nt_ptr(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                      torch.cuda.current_stream().cuda_stream, options, bf16=bf16)
    torch.cuda.synchronize()
    out = Cd.cpu().numpy().view(np.uint16)
    assert np.all(out[:M, N:] == nan), "padding columns of C were written"
    assert np.all(out[M:] == nan), "the row past M was written"
    return np.ascontiguousarray(out[:M, :N])


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("cg,bn", VARIANTS, ids=lambda v: str(v))
def test_forced_small_kernel_matches_oracle(shape, cg, bn):
    M, N, K = shape
    A, B, ref = _reference(M, N, K, False)
    o = g.Options(schedule=5, cta_group=cg, tile_n=bn)
    pl = g.plan(M, N, K, options=o)
    assert (pl["kernel"], pl["cta_group"], pl["tile_n"]) == (1, cg, bn)
    got = _run(A.view(np.uint16), B.view(np.uint16), o)
    check_close(got.view(np.float16), ref, K, f"small kernel {cg}x{bn} {shape}")


@pytest.mark.parametrize("cg,bn", VARIANTS, ids=lambda v: str(v))
def test_forced_small_kernel_integers_bit_exact(cg, bn):
    M, N, K = 300, 520, 1000
    A, B, ref = _reference(M, N, K, True)
    got = _run(A.view(np.uint16), B.view(np.uint16), g.Options(schedule=5, cta_group=cg, tile_n=bn))
    check_bitexact(got.view(np.float16), ref, f"small kernel {cg}x{bn} ints")
    # the same bits on a second call (one tile per cluster, fixed k order)
    again = _run(A.view(np.uint16), B.view(np.uint16), g.Options(schedule=5, cta_group=cg, tile_n=bn))
    assert np.array_equal(got, again)


@pytest.mark.parametrize("cg,bn", [(1, 32), (1, 128), (2, 64)])
@pytest.mark.parametrize("ints", [False, True])
def test_forced_small_kernel_bf16(cg, bn, ints):
    M, N, K = 300, 520, 328
    dist = inputs.I2 if ints else inputs.U
    A = inputs.draw_bf16((M, K), dist, 4301)
    B = inputs.draw_bf16((N, K), dist, 4302)
    got = _run(A, B, g.Options(schedule=5, cta_group=cg, tile_n=bn), bf16=True)
    ref = oracle.gemm_bf16_nt(A, B)
    if ints:
        check_bitexact(got, ref, "bf16 ints")
    else:
        check_close(bf16_to_f64(got), bf16_to_f64(ref), K, "bf16", ulp=ulp_bf16)


@pytest.mark.parametrize("M,N,K,bn", [
    (256, 256, 256, 32),       # 16 tiles
    (64, 64, 64, 32),
    (1024, 1024, 1024, 64),    # 128 tiles
    (1000, 1000, 1000, 64),    # ragged
    (768, 768, 2048, 32),      # 144 tiles: one wave of the SMs
    (128, 4096, 4096, 32),
    (512, 4096, 4096, 128),
])
def test_default_plan_takes_small_kernel_and_matches_oracle(M, N, K, bn):
    pl = g.launch_plan(M, N, K)
    assert (pl["kernel"], pl["cta_group"], pl["tile_n"], pl["workspace_bytes"]) == (1, 1, bn, 0)
    A, B, ref = _reference(M, N, K, False)
    Ad, Bd = to_device(A), to_device(B)
    C, buf = empty_out(M, N, extra_rows=1)
    g.gemm_f16_nt(Ad, Bd, C)
    torch.cuda.synchronize()
    check_close(to_host(C), ref, K, f"default {M}x{N}x{K}")
    assert torch.isnan(buf[M:]).all().item()


def test_stalled_small_kernel_reports_timeout_then_recovers():
    """The documented stall hook with the small kernel: its producer issues no
    copies, so the MMA warp's wait for a filled stage and the epilogue's wait
    for the accumulator run into a 20 ms limit; nothing is written to C."""
    M, N, K = 300, 520, 328
    A, B, ref = _reference(M, N, K, False)
    Ad, Bd = to_device(A), to_device(B)
    for cg in (1, 2):
        C, _ = empty_out(M, N)
        o = g.Options(schedule=5, cta_group=cg, tile_n=64, inject_stall=1, timeout_ns=20_000_000)
        g.gemm_f16_nt(Ad, Bd, C, options=o)
        word = g.device_status()
        assert word & 1, f"watchdog word {word:#x}"
        sites = {s for s in range(1, 8) if word & (1 << (7 + s))}
        assert sites and sites <= {2, 4}, f"unexpected wait sites in {word:#x}"
        assert np.isnan(to_host(C).astype(np.float32)).all(), "C was written by a stalled kernel"
        g.gemm_f16_nt(Ad, Bd, C, options=g.Options(schedule=5, cta_group=cg, tile_n=64))
        torch.cuda.synchronize()
        assert g.device_status() == 0
        check_close(to_host(C), ref, K, f"after the stall, cg{cg}")


def test_small_kernel_captured_and_replayed_with_new_inputs():
    M, N, K = 1024, 1024, 1024
    assert g.launch_plan(M, N, K)["kernel"] == 1
    As = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Bs = torch.empty((N, K), dtype=torch.float16, device="cuda")
    Cs = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    g.gemm_f16_nt(As, Bs, Cs)                      # set-up outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        assert g.launch_plan(M, N, K, stream=s)["kernel"] == 1
        g.gemm_f16_nt(As, Bs, Cs, stream=s)
    for rep in range(2):
        A, B = _operands(M, N, K, True)
        A = np.roll(A, rep, axis=0)
        As.copy_(torch.from_numpy(A))
        Bs.copy_(torch.from_numpy(B))
        Cs.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        check_bitexact(Cs.cpu().numpy(), oracle.gemm_f16_nt(A, B), f"replay {rep + 1}")


@pytest.mark.parametrize("M,N,K,s,ints", [
    (256, 256, 4096, 8, False),     # 16 tiles x 8 pieces of 8 k-blocks
    (256, 256, 4096, 8, True),      # integers: bit-exact, whatever the order of the pieces
    (300, 200, 3000, 4, False),     # 21 ragged tiles x 4 pieces of 11-12 k-blocks
    (512, 512, 8192, 2, False),     # 64 tiles x 2 pieces
    (100, 60, 2000, 4, True),       # 2 tiles of 32 k-blocks: 4 pieces of 8 (8 would leave 4)
])
def test_split_k_small_kernel_matches_oracle(M, N, K, s, ints):
    pl = g.launch_plan(M, N, K)
    assert (pl["kernel"], pl["split_pieces"]) == (1, s) and pl["workspace_bytes"] > 0
    A, B, ref = _reference(M, N, K, ints)
    got = _run(A.view(np.uint16), B.view(np.uint16), None)
    if ints:
        check_bitexact(got.view(np.float16), ref, f"split-K {M}x{N}x{K}")
    else:
        check_close(got.view(np.float16), ref, K, f"split-K {M}x{N}x{K}")
    # the owner adds the pieces in k order: the same bits on every call
    assert np.array_equal(got, _run(A.view(np.uint16), B.view(np.uint16), None))


@pytest.mark.parametrize("cg,bn", [(2, 64), (1, 128), (2, 32)])
def test_split_k_forced_variants_and_bf16(cg, bn):
    M, N, K = 300, 200, 3000
    o = g.Options(schedule=5, cta_group=cg, tile_n=bn)
    pl = g.plan(M, N, K, options=o)
    assert pl["split_pieces"] > 1
    A, B, ref = _reference(M, N, K, False)
    check_close(_run(A.view(np.uint16), B.view(np.uint16), o).view(np.float16), ref, K, f"split-K {cg}x{bn}")
    Ab = inputs.draw_bf16((M, K), inputs.U, 4401)
    Bb = inputs.draw_bf16((N, K), inputs.U, 4402)
    got = _run(Ab, Bb, o, bf16=True)
    check_close(bf16_to_f64(got), bf16_to_f64(oracle.gemm_bf16_nt(Ab, Bb)), K, "split-K bf16", ulp=ulp_bf16)


def test_split_k_small_kernel_under_capture_runs_unsplit():
    """Under stream capture the split is off (its flags are tagged per launch,
    and a replay repeats the launch): one piece a tile, still the oracle's result."""
    M, N, K = 256, 256, 4096
    assert g.launch_plan(M, N, K)["split_pieces"] == 8
    As = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Bs = torch.empty((N, K), dtype=torch.float16, device="cuda")
    Cs = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    g.gemm_f16_nt(As, Bs, Cs)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        pl = g.launch_plan(M, N, K, stream=s)
        g.gemm_f16_nt(As, Bs, Cs, stream=s)
    assert (pl["kernel"], pl["split_pieces"], pl["split_k_off"], pl["workspace_bytes"]) == (1, 1, 1, 0)
    A, B = _operands(M, N, K, True)
    As.copy_(torch.from_numpy(A))
    Bs.copy_(torch.from_numpy(B))
    torch.cuda.synchronize()
    for _ in range(2):
        Cs.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        check_bitexact(Cs.cpu().numpy(), oracle.gemm_f16_nt(A, B), "captured split-K shape")


def test_stalled_split_k_small_kernel_reports_timeout():
    M, N, K = 256, 256, 4096
    A, B, ref = _reference(M, N, K, False)
    Ad, Bd = to_device(A), to_device(B)
    C, _ = empty_out(M, N)
    g.gemm_f16_nt(Ad, Bd, C, options=g.Options(schedule=5, inject_stall=1, timeout_ns=20_000_000))
    word = g.device_status()
    assert word & 1, f"watchdog word {word:#x}"
    sites = {s for s in range(1, 8) if word & (1 << (7 + s))}
    assert sites and sites <= {2, 4, 7}, f"unexpected wait sites in {word:#x}"
    assert np.isnan(to_host(C).astype(np.float32)).all(), "C was written by a stalled kernel"
    g.gemm_f16_nt(Ad, Bd, C)
    torch.cuda.synchronize()
    assert g.device_status() == 0
    check_close(to_host(C), ref, K, "after the stall")
