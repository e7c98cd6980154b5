"""Parity of the bfloat16 entry points (gemm_bf16_nt, gemm_bf16_nt_ex) with the
oracle's bf16 variant: same seeded bf16 inputs, element by element, within
2 bf16 ulps + 1e-4 sqrt(K), bit-exact on small-integer inputs.  C is
pre-filled with a bf16 NaN so unwritten elements show, and padding columns
must come back untouched."""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import lib_for
from tests.tolerance import bf16_to_f64, check_bitexact, check_close, ulp_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402

NAN_BF16 = 0x7FC0


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def dev_bf16(bits: np.ndarray, ld: int | None = None):
    rows, cols = bits.shape
    if ld is None:
        ld = max(cols, 1)
        ld += (-ld) % 8
    buf = np.full((max(rows, 1), ld), NAN_BF16, dtype=np.uint16)
    buf[:rows, :cols] = bits
    t = torch.from_numpy(buf.view(np.int16)).to("cuda:0").view(torch.bfloat16)
    return t[:rows, :cols]


def host_bits(t) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run(A, B, ldc=None, options=None):
    M, N = A.shape[0], B.shape[0]
    Cbuf = dev_bf16(np.full((M, N), NAN_BF16, dtype=np.uint16), ldc)
    g.gemm_bf16_nt(dev_bf16(A), dev_bf16(B), Cbuf, options=options,
                   lib=lib_for(options.cluster_pairs if options is not None else 0))
    torch.cuda.synchronize()
    return host_bits(Cbuf)


@pytest.mark.parametrize("cg,cp", [(2, 1), (1, 1), (2, 2)])
@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 520, 328), (7, 9, 3), (1000, 700, 1000)])
def test_small_shapes(M, N, K, cg, cp):
    A = inputs.draw_bf16((M, K), inputs.U, 401 + M)
    B = inputs.draw_bf16((N, K), inputs.U, 402 + N)
    C = run(A, B, options=g.Options(cta_group=cg, cluster_pairs=cp))
    check_close(bf16_to_f64(C), bf16_to_f64(oracle.gemm_bf16_nt(A, B)), K, f"bf16 {M}x{N}x{K}", ulp=ulp_bf16)


def test_stream_k_and_persistent():
    M, N, K = 1100, 2100, 520
    A = inputs.draw_bf16((M, K), inputs.U, 403)
    B = inputs.draw_bf16((N, K), inputs.U, 404)
    ref = bf16_to_f64(oracle.gemm_bf16_nt(A, B))
    for o in (g.Options(schedule=2, max_clusters=7), g.Options(max_clusters=3, swizzle=3)):
        check_close(bf16_to_f64(run(A, B, options=o)), ref, K, "bf16 stream-K / persistent", ulp=ulp_bf16)


def test_padding_untouched():
    M, N, K = 130, 300, 200
    A = inputs.draw_bf16((M, K), inputs.U, 405)
    B = inputs.draw_bf16((N, K), inputs.U, 406)
    Cbuf_np = np.full((M, N + 20), NAN_BF16, dtype=np.uint16)
    Cd = dev_bf16(Cbuf_np)
    g.gemm_bf16_nt(dev_bf16(A), dev_bf16(B), Cd[:, :N])
    torch.cuda.synchronize()
    out = host_bits(Cd)
    assert np.all(out[:, N:] == NAN_BF16)
    check_close(bf16_to_f64(out[:, :N]), bf16_to_f64(oracle.gemm_bf16_nt(A, B)), K, "bf16 pitched",
                ulp=ulp_bf16)


def test_ragged_integers_bit_exact():
    M, N, K = 4000, 3000, 5000
    A = inputs.draw_bf16((M, K), inputs.I2, 407)
    B = inputs.draw_bf16((N, K), inputs.I2, 408)
    check_bitexact(run(A, B).view(np.float16), oracle.gemm_bf16_nt(A, B).view(np.float16), "bf16 int ragged")


def test_8192_sampled():
    M = N = K = 8192
    A = inputs.draw_bf16((M, K), inputs.U, 409)
    B = inputs.draw_bf16((N, K), inputs.U, 410)
    C = run(A, B)
    assert not np.any(C == NAN_BF16)
    rng = np.random.default_rng(1)
    rows = np.concatenate([rng.integers(0, M, 2000), [0, M - 1, 0, M - 1]])
    cols = np.concatenate([rng.integers(0, N, 2000), [0, 0, N - 1, N - 1]])
    ref = oracle.gemm_bf16_nt_points(A, B, rows, cols)
    check_close(bf16_to_f64(C[rows, cols]), bf16_to_f64(ref), K, "bf16 8192 sampled", ulp=ulp_bf16)


@pytest.mark.parametrize("a_layout,b_layout", [(0, 1), (1, 1)])
def test_bf16_operand_layouts(a_layout, b_layout):
    M, N, K = 600, 700, 520
    A = inputs.draw_bf16((M, K), inputs.U, 411)
    B = inputs.draw_bf16((N, K), inputs.U, 412)
    A_st = np.ascontiguousarray(A.T) if a_layout else A
    B_st = np.ascontiguousarray(B.T) if b_layout else B
    C = g.gemm_bf16_nt(dev_bf16(A_st), dev_bf16(B_st), a_layout=a_layout, b_layout=b_layout)
    torch.cuda.synchronize()
    check_close(bf16_to_f64(host_bits(C)), bf16_to_f64(oracle.gemm_bf16_nt(A, B)), K,
                f"bf16 layout A{a_layout} B{b_layout}", ulp=ulp_bf16)
