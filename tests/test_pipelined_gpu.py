"""GPU tests of the _pipelined verify calls: x, a and b of a (request, layer)
are read only once its flag in x_ready is set, by a copy queued behind the
rows. Same bytes as the plain call, whether the flags were set before the
launch or land while it runs; a flag that nothing sets ends the bounded
wait with GDN_DEV_SCHED instead of a hang."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_layer_vs_oracle, ensure_built
from speculative_decode_hybrid_gb300 import gdnspec as G
from speculative_decode_hybrid_gb300 import workloads as W
from speculative_decode_hybrid_gb300.pipeline import SpecStep

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    ensure_built()


def _same(a, b):
    for name in ("out", "ssm_ckpt", "conv_ckpt"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


@pytest.mark.parametrize("wid,layers", [(2, 3), (3, 3), (1, None), (4, 2)])
def test_pipelined_with_flags_set_equals_plain(wid, layers):
    """Every flag set before the launch: the plain call's bytes (one-layer
    launches, multi-layer launches with work stealing, trees, batch 16)."""
    wl = W.make_workload(wid, seed=33, **({} if layers is None else {"layers": layers}))
    a, b = SpecStep(wl), SpecStep(wl)
    a.verify()
    b.x_ready.fill_(1)
    b.verify(x_ready=b.x_ready)
    torch.cuda.synchronize()
    _same(a, b)
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("wid,layers", [(2, 4), (3, 4), (4, 2)])
def test_pipelined_waits_for_flags_landing_during_the_launch(wid, layers):
    """The inputs and their flags are copied on another stream behind a
    large host-to-device copy (a few hundred microseconds), after the verify
    has been queued: the kernel waits for each item's flag and gives the
    plain call's bytes, with no status bit set. Batch 16 runs more items than
    CTAs (work stealing): a CTA whose next item has not landed when it takes
    it stages that item after the current one's recurrence."""
    wl = W.make_workload(wid, seed=34, layers=layers)
    ref = SpecStep(wl)
    ref.verify()
    st = SpecStep(wl)
    host = {n: getattr(st, n).cpu().pin_memory() for n in ("x", "a", "b")}
    for n in ("x", "a", "b"):
        getattr(st, n).zero_()  # the verify must not see these before its flags
    ballast_h = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    ballast_d = torch.empty_like(ballast_h, device="cuda")
    ones = st._ones
    torch.cuda.synchronize()
    copy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    with torch.cuda.stream(copy):
        ballast_d.copy_(ballast_h, non_blocking=True)  # the DMA queue is busy for a while
        Y = wl.shape.layers
        for b_ in range(wl.shape.batch):
            for y in range(Y):
                for n in ("x", "a", "b"):
                    getattr(st, n)[b_, y].copy_(host[n][b_, y], non_blocking=True)
                st.x_ready.view(-1)[b_ * Y + y:b_ * Y + y + 1].copy_(ones[b_ * Y + y:b_ * Y + y + 1],
                                                                      non_blocking=True)
    st.verify(stream=main, x_ready=st.x_ready)  # queued while the copies are still in flight
    torch.cuda.synchronize()
    _same(ref, st)
    assert int(st.dev_status.item()) == 0
    check_layer_vs_oracle(st, wl, 0, min(2, layers - 1))


def test_pipelined_wait_gives_up_on_a_flag_nothing_sets():
    """x_ready all zero and nothing to set it: the bounded wait of every item
    ends (about a quarter second) and the kernel sets GDN_DEV_SCHED; the
    context stays usable (a plain verify afterwards gives its bytes)."""
    wl = W.make_workload(1, seed=35)
    st = SpecStep(wl)
    st.verify(x_ready=st.x_ready)
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) & G.GDN_DEV_SCHED
    a, b = SpecStep(wl), SpecStep(wl)
    a.verify()
    b.verify()
    torch.cuda.synchronize()
    _same(a, b)
    assert int(b.dev_status.item()) == 0


@pytest.mark.parametrize("tree", [False, True])
def test_pipelined_on_the_fallback_kernel(tree):
    """An x that is not 16-byte aligned takes the one-item-per-CTA kernel, whose
    CTAs wait for their item's flag at entry: with the rows and flags landing
    behind a long copy, the same bytes as the plain call (which runs the
    staged kernel on an aligned x)."""
    wl = W.make_workload(3 if tree else 2, seed=36, layers=3)
    ref = SpecStep(wl)
    ref.verify()
    st = SpecStep(wl)
    host = {n: getattr(st, n).cpu().pin_memory() for n in ("x", "a", "b")}
    shifted = torch.empty(st.x.numel() + 8, dtype=st.x.dtype, device="cuda")
    st.x = shifted[1:1 + st.x.numel()].view(st.x.shape)  # a 2-byte offset
    assert st.x.data_ptr() % 16 != 0
    for n in ("x", "a", "b"):
        getattr(st, n).zero_()
    ballast_h = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    ballast_d = torch.empty_like(ballast_h, device="cuda")
    torch.cuda.synchronize()
    copy = torch.cuda.Stream()
    with torch.cuda.stream(copy):
        ballast_d.copy_(ballast_h, non_blocking=True)
        Y = wl.shape.layers
        for y in range(Y):
            for n in ("x", "a", "b"):
                getattr(st, n)[0, y].copy_(host[n][0, y], non_blocking=True)
            st.x_ready.view(-1)[y:y + 1].copy_(st._ones[y:y + 1], non_blocking=True)
    st.verify(stream=torch.cuda.current_stream(), x_ready=st.x_ready)
    torch.cuda.synchronize()
    _same(ref, st)
    assert int(st.dev_status.item()) == 0
