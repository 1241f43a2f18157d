"""Failure detection without a GPU fault.

Every mbarrier wait in the GEMM kernel is bounded. A test-only switch makes
the first CTA of the next GEMM launch withhold one operand load, so the MMA
warp's wait on that stage runs out (after a 100 ms limit set for the test).
In a paired launch (the 2-SM MMA, cta_group::2) each CTA of the pair loads
its own half of the operands, and both halves count on one barrier of the
even CTA, so a half withheld by either CTA starves the pair's MMA; no TMA
multicast is involved.
The kernel then raises its abort flag, drains the copies and MMAs it started,
frees its tensor memory and returns; the host reads TP_ERR_TIMEOUT from
tp_get_error(), and the next launch on the same context computes correctly.
Nothing here traps, faults or hangs the GPU: the "failure" is a wait that
nobody satisfies, and every wait has a time limit.
"""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import tp_oracle as O
from tests._util import TOL_BF16, assert_close, dev, f64

pytestmark = pytest.mark.gpu

tpl = pytest.importorskip("tensor_transformer_linear_tma_b300")

TP_ERR_TIMEOUT = 8


@pytest.fixture
def short_wait_limit():
    assert tpl.tp_get_error() == 0
    tpl.tp_debug_set_wait_limit_ns(100_000_000)
    yield
    tpl.tp_debug_inject(0)
    tpl.tp_debug_set_wait_limit_ns(2_000_000_000)
    tpl.tp_get_error()


@pytest.mark.parametrize("path", ["whole_tiles", "cluster_pairs", "cluster_pairs_odd", "weight_streaming"])
def test_expired_wait_is_reported_and_context_survives(short_wait_limit, path):
    # 300 tokens: 3 token blocks, single CTAs; 512 tokens: 4 blocks, CTA pairs
    # on the 2-SM MMA, each CTA loading its own operand half (the withheld load
    # starves the pair's MMA). Withheld by the even CTA, the even CTA arms the
    # odd CTA's half of that stage alone when it drains; withheld by the odd
    # CTA, it counts the missing half as arrived. Either way the odd CTA
    # leaves only once the even CTA has seen every copy it started land.
    T = {"whole_tiles": 300, "cluster_pairs": 512, "cluster_pairs_odd": 512, "weight_streaming": 8}[path]
    K, N, tp = 256, 2 * 1024, 2
    X, W = S.normal(101, (T, K)), S.normal(102, (K, N), 0.05)
    Sc = tpl.tp_shard_weights(dev(W), tp, "col")
    ws = None
    if path == "weight_streaming":  # T <= 64 with a workspace: split tiles, stream-K schedule
        ws = torch.empty(tpl.tp_gemm_workspace_bytes(T, Sc), dtype=torch.uint8, device="cuda")
        assert ws.numel() > 0
    ref = np.stack(O.column_parallel(f64(X), f64(W), tp))
    Xd = dev(X)
    torch.cuda.synchronize()

    tpl.tp_debug_inject(2 if path == "cluster_pairs_odd" else 1)
    tpl.tp_column_linear(Xd, Sc, workspace=ws)
    assert tpl.tp_get_error() == TP_ERR_TIMEOUT

    Y = tpl.tp_column_linear(Xd, Sc, workspace=ws)   # same context, switch consumed
    assert tpl.tp_get_error() == 0
    assert_close(Y, ref, TOL_BF16, f"after a timeout ({path})")
