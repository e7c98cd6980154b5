"""The stream-K workspace: reserved once per device at set-up, never allocated
per call, shared by concurrent streams through slots, and its absence visible.

A stream-K launch takes one of the slots reserved at the device's set-up; the
call orders its stream after the slot's previous user.  These tests check that
no call allocates device memory, that many stream-K calls spread over more
streams than there are slots all give the oracle's result, and that with no
slots (GEMM_F16_NT_WORKSPACE_SLOTS=0, in a child process) the plan reports the
fall-back and the result is still right.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, to_device, to_host
from tests.tolerance import check_bitexact, check_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0


def test_slots_reserved_and_no_allocation_per_call():
    M, N, K = 4096, 4096, 4096          # 256 tiles on 76 pairs: stream-K by default
    pl = g.launch_plan(M, N, K)
    assert pl["sk_tiles"] > 0 and pl["split_k_off"] == 0
    ws = g.device_workspace()
    assert ws["slots"] == 4 and ws["bytes_per_slot"] >= pl["workspace_bytes"]
    A = inputs.draw((M, K), inputs.I2, 3101)
    B = inputs.draw((N, K), inputs.I2, 3102)
    Ad, Bd = to_device(A), to_device(B)
    outs = [empty_out(M, N)[0] for _ in range(3)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for C in outs:
        g.gemm_f16_nt(Ad, Bd, C)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the calls"
    ref = oracle.gemm_f16_nt(A, B)
    for C in outs:
        check_bitexact(to_host(C), ref, "stream-K through a reserved slot")


def test_capture_reports_split_off():
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    A = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    C = torch.empty((4096, 4096), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(A, A, C)                          # set-up outside the capture
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        pl = g.launch_plan(4096, 4096, 4096, stream=s)
        g.gemm_f16_nt(A, A, C, stream=s)
    assert (pl["sk_tiles"], pl["split_k_off"]) == (0, 1)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.count_nonzero(C).item() == 0


def test_more_concurrent_streams_than_slots():
    """Ten stream-K calls on six unordered streams (four slots): calls that land
    on a busy slot wait for it, and every result is the oracle's, bit for bit."""
    M, N, K = 1100, 2100, 520
    o = g.Options(schedule=2, max_clusters=7)       # 45 tiles on 7 pairs, split in k
    assert g.launch_plan(M, N, K, options=o)["sk_tiles"] > 0
    streams = [torch.cuda.Stream() for _ in range(6)]
    cases = []
    for i in range(10):
        A = inputs.draw((M, K), inputs.I2, 3200 + i)
        B = inputs.draw((N, K), inputs.I2, 3300 + i)
        cases.append((A, B, to_device(A), to_device(B), empty_out(M, N)[0]))
    torch.cuda.synchronize()
    for i, (_, _, Ad, Bd, C) in enumerate(cases):
        g.gemm_f16_nt(Ad, Bd, C, stream=streams[i % 6], options=o)
    torch.cuda.synchronize()
    for i, (A, B, _, _, C) in enumerate(cases):
        check_bitexact(to_host(C), oracle.gemm_f16_nt(A, B), f"call {i}")


def test_without_workspace_slots_the_split_is_off_and_visible():
    code = textwrap.dedent("""
        import json, sys
        sys.path.insert(0, %r)
        import numpy as np, torch
        import dense_fp16_gemm_gb300 as g
        import oracle
        from dense_fp16_gemm_gb300 import inputs
        from tests.tolerance import check_close
        M, N, K = 4096, 4096, 4096
        pl = g.launch_plan(M, N, K)
        ws = g.device_workspace()
        A = inputs.draw((M, K), inputs.U, 3401)
        B = inputs.draw((N, K), inputs.U, 3402)
        Ad = torch.from_numpy(A).cuda(); Bd = torch.from_numpy(B).cuda()
        C = g.gemm_f16_nt(Ad, Bd)
        torch.cuda.synchronize()
        check_close(C.cpu().numpy(), oracle.gemm_f16_nt(A, B), K, "no workspace")
        print(json.dumps({"plan": pl, "ws": ws, "status": g.device_status()}))
    """ % ROOT)
    env = dict(os.environ, GEMM_F16_NT_WORKSPACE_SLOTS="0")
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    import json
    out = json.loads(res.stdout.strip().splitlines()[-1])
    assert out["ws"] == {"slots": 0, "bytes_per_slot": 0}
    assert (out["plan"]["sk_tiles"], out["plan"]["split_k_off"]) == (0, 2)
    assert out["status"] == 0
