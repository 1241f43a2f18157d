"""tp_mlp_block_static: the MLP block for callers that cannot allocate device
memory (a plug-in whose host process owns the device-memory budget, a path
where the driver's allocator must not be entered). Its workspace is the
library's static device array instead of a caller buffer.

The entry point is called through the C ABI (ctypes, no Python wrapper) two
times in a row and compared with the existing tp_mlp_block, which takes a
caller workspace, within the bf16 tolerance of the other tests
(max|a - b| <= 2e-2 * RMS), and with the oracle. Requests whose workspace
would exceed the static array are refused with TP_ERR_WORKSPACE before
anything is launched. The second call must leave the device's free memory
exactly as it found it (a cudaMalloc inside would take at least one 2 MiB
page). This file is collected last so that a failure here
cannot hide the other tests' results; it also passes on its own in a fresh
process (the first call on the device performs the one-time address lookup).
"""
import ctypes

import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, assert_close, dev, f64, host

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")

TP_ERR_WORKSPACE = 6
ACT_SWIGLU = 4
TP_BF16 = 1


def call_static(X, T, Sg, Su, Sd, R, Y):
    """Direct C-ABI call of tp_mlp_block_static."""
    f = tpl.lib.tp_mlp_block_static
    return f(ctypes.c_void_p(X.data_ptr()), T, Sg.ref(), Su.ref(), Sd.ref(), None, None, None,
             ctypes.c_void_p(R.data_ptr()), ACT_SWIGLU, TP_BF16, ctypes.c_void_p(Y.data_ptr()),
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("T,H,I,tp", [(8, 512, 8 * 136, 8), (64, 1024, 8 * 344, 8), (200, 256, 2 * 344, 2)])
def test_static_workspace_matches_caller_workspace(T, H, I, tp):
    d = S.swiglu_mlp(T, H, I, seeds=(111, 112, 113, 114))
    R = S.normal(115, (T, H))
    Sg, Su = (tpl.tp_shard_weights(dev(d[k]), tp, "col") for k in ("Wg", "Wu"))
    Sd = tpl.tp_shard_weights(dev(d["Wd"]), tp, "row")
    X, Rd = dev(d["X"]), dev(R)
    assert tpl.tp_mlp_workspace_bytes(T, H, I, tp, torch.bfloat16) <= tpl.TP_STATIC_WORKSPACE_BYTES
    Y_ref = tpl.tp_mlp_block(X, Sg, Sd, W_up=Su, residual=Rd, act="swiglu")   # caller workspace
    _, oracle_Y = O.mlp_block(f64(d["X"]), f64(d["Wg"]), f64(d["Wd"]), tp, "swiglu", W_up=f64(d["Wu"]),
                              residual=f64(R))
    for call in range(2):  # two calls in a row share (and reuse) the static array
        Y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert call_static(X, T, Sg, Su, Sd, Rd, Y) == 0
        torch.cuda.synchronize()
        if call == 1:  # after the first call, a call takes no device memory at all
            assert torch.cuda.mem_get_info()[0] == free_before, "the call changed free device memory"
        assert tpl.tp_get_error() == 0
        assert_close(Y, host(Y_ref), TOL_BF16, f"static vs caller workspace, call {call}")
        assert_close(Y, oracle_Y, TOL_BF16, f"static vs oracle, call {call}")


def test_static_workspace_refuses_oversized_requests():
    T, H, I, tp = 2048, 256, 8 * 1376, 8   # Hs alone is 45 MB > 32 MiB
    assert tpl.tp_mlp_workspace_bytes(T, H, I, tp, torch.bfloat16) > tpl.TP_STATIC_WORKSPACE_BYTES
    Wg = torch.zeros((H, I), dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros((I, H), dtype=torch.bfloat16, device="cuda")
    Sg = tpl.tp_shard_weights(Wg, tp, "col")
    Sd = tpl.tp_shard_weights(Wd, tp, "row")
    X = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    Y = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
    assert call_static(X, T, Sg, Sg, Sd, Y, Y) == TP_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all()), "a refused call must launch nothing"
    assert np.isfinite(host(Y)).all()
