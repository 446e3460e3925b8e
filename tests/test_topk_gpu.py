"""spec_topk (draft-side top-k over the vocabulary) against the oracle:
indices and values bit-exact, in the greedy order."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ensure_built
from speculative_decode_hybrid_gb300 import gdnspec as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def topk_gpu(logits, k, ws=None):
    rows, V = logits.shape
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(dev)
    idx = torch.full((rows, k), -3, dtype=torch.int32, device=dev)
    val = torch.zeros((rows, k), dtype=torch.float32, device=dev)
    wsb = G.spec_topk_workspace_bytes(rows, k)
    if ws is None:
        ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
    ds = torch.zeros((1,), dtype=torch.int32, device=dev)
    G.spec_topk(rows, V, k, lg, idx, val, ws, wsb, ds)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy(), int(ds.item())


def check(logits, k, ws=None):
    idx, val, ds = topk_gpu(logits, k, ws)
    for r in range(logits.shape[0]):
        oi, ov = oracle.topk_f32(logits[r], k)
        np.testing.assert_array_equal(idx[r], oi)
        np.testing.assert_array_equal(val[r].view(np.uint32), ov.view(np.uint32))
    return ds


@pytest.mark.parametrize("k", [1, 8, 22, 32])
def test_topk_qwen_vocab(k):
    g = np.random.default_rng(k)
    logits = g.standard_normal((5, 151936)).astype(np.float32)
    assert check(logits, k) == 0


@pytest.mark.parametrize("V", [32, 33, 1001, 4096, 70001])
def test_topk_ties_and_sizes(V):
    g = np.random.default_rng(V)
    logits = g.integers(-3, 4, (3, V)).astype(np.float32)     # many ties
    check(logits, min(32, V))
    check(logits, min(5, V))


def test_topk_nan_signed_zero_and_infinities():
    g = np.random.default_rng(5)
    logits = g.standard_normal((2, 9000)).astype(np.float32)
    logits[0, [100, 7000, 50]] = np.nan
    logits[0, [1, 2, 3]] = np.inf
    logits[1, :] = 0.0
    logits[1, ::2] = -0.0
    logits[1, 8999] = -np.inf
    ds = check(logits, 10)
    assert ds & G.GDN_DEV_NAN_LOGIT


def test_topk_many_rows_and_workspace_reuse():
    g = np.random.default_rng(9)
    dev = torch.device("cuda")
    wsb = G.spec_topk_workspace_bytes(400, 32)
    ws = torch.zeros((wsb,), dtype=torch.uint8, device=dev)
    for rows, V, k in ((368, 151936, 16), (3, 5000, 32), (400, 2048, 7), (70, 9000, 3)):
        logits = g.standard_normal((rows, V)).astype(np.float32)
        idx, val, _ = topk_gpu(logits, k, ws)
        for r in (0, rows // 2, rows - 1):
            oi, _ = oracle.topk_f32(logits[r], k)
            np.testing.assert_array_equal(idx[r], oi)
        assert int(ws.count_nonzero().item()) == 0   # every call leaves it zero-filled
