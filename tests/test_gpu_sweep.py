"""A seeded sweep of random configurations through the C ABI, each checked
element by element against the oracle.

Every case draws its sizes (log-uniform in 1..2600), operand layouts, padded
row pitches, cluster shape, schedule, operand type (fp16 or bf16), accumulator
(fp32, or fp16 for some fp16 cases) and input distribution from one fixed
seed, so the sweep is the same on every run.  Padding columns of A and B hold
NaN (a read of them would poison the result); C's padding columns and an extra
row past M must come back untouched.

Bars: small-integer inputs with fp32 accumulation are bit-exact; other fp32
cases are within 2 ulps of the output format + 1e-4·sqrt(K); fp16-accumulator
cases follow the oracle's per-16-k model (at least 98 % of outputs identical,
every output within 8 fp16 ulps of the rms output magnitude).
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import lib_for
from tests.tolerance import bf16_to_f64, check_bitexact, check_close, ulp_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402

NAN = {"f16": 0x7E00, "bf16": 0x7FC0}


def _configs(n=48, seed=20261202, schedules=(0, 0, 1, 2, 3), mn_max=2600, k_min=1):
    rng = np.random.default_rng(seed)
    size = lambda hi=2600: int(np.clip(np.round(np.exp(rng.uniform(0.0, np.log(float(hi))))), 1, hi))
    out = []
    for i in range(n):
        dtype = "bf16" if rng.random() < 0.3 else "f16"
        cg = 1 if rng.random() < 0.25 else 2
        cp = 0 if cg == 1 else int(rng.choice([0, 0, 1, 2]))
        out.append(dict(
            i=i, M=size(mn_max), N=size(mn_max), K=max(size(), k_min), dtype=dtype,
            acc16=dtype == "f16" and rng.random() < 0.2,
            a_layout=int(rng.integers(0, 2)), b_layout=int(rng.integers(0, 2)),
            cg=cg, cp=cp, schedule=int(rng.choice(list(schedules))),
            pad=[int(rng.choice([0, 8, 64])) for _ in range(3)],
            ints=rng.random() < 0.3))
    return out


# the first 48 as before; 24 more that force split pieces (every option and
# type with each tile cut along k, wherever the tiles leave room for two pieces)
CASES = _configs() + [dict(c, i=100 + c["i"]) for c in _configs(24, 20261204, (4,), mn_max=1200, k_min=200)]


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def _bits(x, dtype):
    """16-bit patterns of a float16 array (fp16) or of a bf16 uint16 array."""
    return x.view(np.uint16) if dtype == "f16" else x


def _device(bits, ld, nan):
    rows, cols = bits.shape
    buf = np.full((max(rows, 1), ld), nan, dtype=np.uint16)
    buf[:rows, :cols] = bits
    return torch.from_numpy(buf.view(np.int16)).cuda()


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"{c['i']}-{c['M']}x{c['N']}x{c['K']}-{c['dtype']}"
                         f"{'-acc16' if c['acc16'] else ''}-L{c['a_layout']}{c['b_layout']}-cg{c['cg']}"
                         f"cp{c['cp']}-s{c['schedule']}{'-int' if c['ints'] else ''}")
def test_random_configuration(c):
    M, N, K, dt = c["M"], c["N"], c["K"], c["dtype"]
    dist = inputs.I2 if c["ints"] else inputs.U
    draw = inputs.draw if dt == "f16" else inputs.draw_bf16
    A = draw((M, K), dist, 5000 + c["i"])
    B = draw((N, K), dist, 6000 + c["i"])
    a_st = np.ascontiguousarray(_bits(A, dt).T) if c["a_layout"] else _bits(A, dt)
    b_st = np.ascontiguousarray(_bits(B, dt).T) if c["b_layout"] else _bits(B, dt)
    r8 = lambda v: v + (-v) % 8
    lda = r8(a_st.shape[1]) + c["pad"][0]
    ldb = r8(b_st.shape[1]) + c["pad"][1]
    ldc = r8(N) + c["pad"][2]
    Ad, Bd = _device(a_st, lda, NAN[dt]), _device(b_st, ldb, NAN[dt])
    Cd = _device(np.full((M + 1, ldc), NAN[dt], dtype=np.uint16), ldc, NAN[dt])
    o = g.Options(cta_group=c["cg"], cluster_pairs=c["cp"], schedule=c["schedule"],
                  a_layout=c["a_layout"], b_layout=c["b_layout"], accumulate=int(c["acc16"]))
    g.gemm_f16_nt_ptr(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                      torch.cuda.current_stream().cuda_stream, o, bf16=dt == "bf16", lib=lib_for(c["cp"]))
    torch.cuda.synchronize()
    out = Cd.cpu().numpy().view(np.uint16)
    assert np.all(out[:M, N:] == NAN[dt]), "padding columns of C were written"
    assert np.all(out[M:] == NAN[dt]), "the row past M was written"
    got = np.ascontiguousarray(out[:M, :N])
    if dt == "bf16":
        ref = oracle.gemm_bf16_nt(A, B)
        if c["ints"]:
            check_bitexact(got, ref, "bf16 ints")
        else:
            check_close(bf16_to_f64(got), bf16_to_f64(ref), K, "bf16", ulp=ulp_bf16)
    elif c["acc16"]:
        ref = oracle.gemm_f16_nt_acc16(A, B).astype(np.float64)
        C = got.view(np.float16).astype(np.float64)
        assert np.mean(C == ref) >= 0.98
        rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
        if rms > 0:
            assert np.abs(C - ref).max() <= 8 * 2.0 ** (np.floor(np.log2(rms)) - 10)
    else:
        ref = oracle.gemm_f16_nt(A, B)
        if c["ints"]:
            check_bitexact(got.view(np.float16), ref, "f16 ints")
        else:
            check_close(got.view(np.float16), ref, K, "f16")
