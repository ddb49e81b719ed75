"""ts_hc_call_noalloc (no workspace, nothing allocated) against ts_hc_call.

Some callers cannot allocate device memory when they run the call: real-time
loops that cannot afford the implicit synchronisation an allocation may cause,
and hosts that give the library a fixed memory budget and no allocator. For them the
library keeps the call's scratch in a device array of its own. These tests call
that entry point through the C ABI twice in a row -- first 128 tokens (the
tensor-core path), then one token (the CUDA-core path), so the second call runs
over the first call's leftovers in the shared array -- and compare both results
with ts_hc_call on the same inputs, within the parity tolerances used
everywhere else. This file is collected last so that a failure here comes
after every other test has run.
"""
import pytest
import torch

from hyper_connection_residual_call_gb300 import binding as B
from hyper_connection_residual_call_gb300 import inputs
from gpu_common import check_bf16, check_fp32, require_gpu

pytestmark = pytest.mark.gpu
EPS = 1e-6
H, C, L = 2560, 4, 320


def _inputs(M, seed):
    w = inputs.make_hc_weights(H, C, L, seed).to("cuda")
    raw = inputs.make_residual(M, H, C, seed).cuda()
    return w, raw


def _noalloc(raw, w):
    """Outputs are the caller's (allocated here by the test); the call itself allocates nothing."""
    M = raw.shape[0]
    mixed = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    gates = torch.empty((M, C), dtype=torch.float32, device="cuda")
    st = B.ts_hc_call_noalloc(raw.data_ptr(), w.g.data_ptr(), B.weight_struct(w.down), B.weight_struct(w.up),
                              B.weight_struct(w.inject), mixed.data_ptr(), gates.data_ptr(), C, M, H, C, L,
                              EPS, torch.cuda.current_stream().cuda_stream)
    assert st == B.TS_OK, B.ts_hc_last_error()
    return mixed, gates


def test_noalloc_matches_call_on_two_calls_in_a_row():
    require_gpu()
    cases = [_inputs(128, 501), _inputs(1, 502)]
    got = [_noalloc(raw, w) for w, raw in cases]   # two calls back to back on one stream
    want = [B.hc_call(raw, w, H=H, C=C, eps=EPS) for w, raw in cases]
    torch.cuda.synchronize()
    for (gm, gg), (wm, wg), (w, raw) in zip(got, want, cases):
        M = raw.shape[0]
        check_bf16(gm, wm.double().cpu().numpy(), f"no-alloc mixed, M={M}")
        check_fp32(gg, wg.double().cpu().numpy(), f"no-alloc gates, M={M}")
    assert B.device_status() == B.TS_OK


def test_noalloc_allocates_nothing():
    """After a first call (which looks up the array's address), a call changes
    neither torch's allocated bytes nor the device's free memory."""
    require_gpu()
    w, raw = _inputs(16, 504)
    mixed = torch.empty((16, H), dtype=torch.bfloat16, device="cuda")
    gates = torch.empty((16, C), dtype=torch.float32, device="cuda")
    args = (raw.data_ptr(), w.g.data_ptr(), B.weight_struct(w.down), B.weight_struct(w.up), B.weight_struct(w.inject),
            mixed.data_ptr(), gates.data_ptr(), C, 16, H, C, L, EPS, torch.cuda.current_stream().cuda_stream)
    assert B.ts_hc_call_noalloc(*args) == B.TS_OK, B.ts_hc_last_error()
    torch.cuda.synchronize()
    torch_bytes, (free, _) = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()
    assert B.ts_hc_call_noalloc(*args) == B.TS_OK, B.ts_hc_last_error()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_bytes
    assert torch.cuda.mem_get_info()[0] == free


def _first_token_count_over_the_scratch():
    lo, hi = 1, 1 << 20
    while lo < hi:
        mid = (lo + hi) // 2
        if B.ts_hc_workspace_bytes(mid, H, C, L) > B.TS_HC_STATIC_SCRATCH_BYTES:
            hi = mid
        else:
            lo = mid + 1
    return lo


def test_noalloc_refuses_more_tokens_than_its_scratch_holds():
    require_gpu()
    M = _first_token_count_over_the_scratch()  # 1374 at this shape
    assert B.ts_hc_workspace_bytes(M, H, C, L) > B.TS_HC_STATIC_SCRATCH_BYTES
    assert B.ts_hc_workspace_bytes(M - 1, H, C, L) <= B.TS_HC_STATIC_SCRATCH_BYTES
    w, raw = _inputs(2, 503)
    st = B.ts_hc_call_noalloc(raw.data_ptr(), w.g.data_ptr(), B.weight_struct(w.down), B.weight_struct(w.up),
                              B.weight_struct(w.inject), raw.data_ptr(), raw.data_ptr(), C, M, H, C, L, EPS,
                              torch.cuda.current_stream().cuda_stream)
    assert st == B.TS_ERR_WORKSPACE
    assert "static scratch holds" in B.ts_hc_last_error()
