"""gemm_f16_nt_noalloc: C = A·Bᵀ without taking any device memory.

Some callers cannot let a library allocate device memory at all: their own
allocator has reserved the memory up front, or the call sits in a
latency-critical loop.  For them the library keeps the stream-K scratch in a
fixed 20 MiB array compiled into it.  This file checks, through the C ABI, that
the entry point gives the oracle's product (within the parity tolerance, bit
for bit on small-integer inputs) and the same product as gemm_f16_nt, on two
calls in a row, the second one finding the first one's leftovers in the shared
scratch, and that device free memory does not move.  A call made while its
stream is capturing is planned without the split, as gemm_f16_nt's is; the
last case checks that such a call, replayed with new inputs, still matches the
oracle.  It is named to be collected last.
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, to_device, to_host
from tests.tolerance import check_bitexact, check_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


def _call(fn, A, B, C, stream):
    M, K = A.shape
    N = B.shape[0]
    return fn(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
              C.stride(0), stream)


@pytest.mark.parametrize("M,N,K,uses_scratch,ints", [
    (1024, 1024, 12288, True, False),    # 16 pair tiles, each in 4 split pieces over 64 pairs
    (6144, 4096, 4096, True, False),     # 384 tiles: last wave 4/76 full, deep k: stream-K part
    (1024, 1024, 12288, True, True),     # integers: exact, whatever the summation order
    (256, 256, 4096, True, True),        # the small-problem kernel's split-K: 16 tiles x 8 pieces
    (300, 520, 328, False, False),       # the small-problem kernel: no scratch needed
    (1024, 1024, 1024, False, True),     # the same, 128 tiles of 128 x 64, integers
])
def test_noalloc_matches_oracle_and_gemm_f16_nt_on_two_calls(M, N, K, uses_scratch, ints):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = g.library()
    pl = g.launch_plan(M, N, K)
    assert (pl["workspace_bytes"] > 0) == uses_scratch
    dist = inputs.I2 if ints else inputs.U
    A = inputs.draw((M, K), dist, 301 + M)
    B = inputs.draw((N, K), dist, 302 + N)
    Ad, Bd = to_device(A), to_device(B)
    stream = torch.cuda.current_stream().cuda_stream

    ref, _ = empty_out(M, N)
    assert _call(lib.gemm_f16_nt, Ad, Bd, ref, stream) == 0
    outs = [empty_out(M, N)[0] for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for C in outs:
        assert _call(lib.gemm_f16_nt_noalloc, Ad, Bd, C, stream) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the calls"
    assert g.device_status() == 0
    expect = to_host(ref)
    want = oracle.gemm_f16_nt(A, B)
    for i, C in enumerate(outs):
        got = to_host(C)
        if ints:
            check_bitexact(got, want, f"gemm_f16_nt_noalloc call {i + 1} vs oracle")
        else:
            check_close(got, want, K, f"gemm_f16_nt_noalloc call {i + 1} vs oracle")
        check_close(got, expect, K, f"gemm_f16_nt_noalloc call {i + 1} vs gemm_f16_nt")


def test_noalloc_call_under_capture_replays_with_new_inputs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = g.library()
    M, N, K = 1024, 1024, 12288                   # split in k when called directly
    assert g.launch_plan(M, N, K)["workspace_bytes"] > 0
    Ad = torch.empty((M, K), dtype=torch.float16, device="cuda")
    Bd = torch.empty((N, K), dtype=torch.float16, device="cuda")
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        assert g.launch_plan(M, N, K, stream=s)["split_k_off"] == 1
        assert _call(lib.gemm_f16_nt_noalloc, Ad, Bd, C, s.cuda_stream) == 0
    for rep in range(2):
        A = inputs.draw((M, K), inputs.I2, 311 + rep)
        B = inputs.draw((N, K), inputs.I2, 312 + rep)
        Ad.copy_(torch.from_numpy(A))
        Bd.copy_(torch.from_numpy(B))
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        check_bitexact(to_host(C), oracle.gemm_f16_nt(A, B), f"captured noalloc call, replay {rep + 1}")
    assert g.device_status() == 0
