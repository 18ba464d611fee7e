"""Bounds and status checks on the GPU: outputs are written exactly in place.

Each output lives inside a larger buffer whose guard bytes before and after it
hold a known pattern; after the call the guards must be unchanged. This is the
bounds check used instead of a memory sanitizer.
"""
import pytest
import torch

from depth_wise_attention_attnres_gb300 import binding as ar
from depth_wise_attention_attnres_gb300 import inputs
from tests._gpu import dev

pytestmark = pytest.mark.gpu
GUARD = 4096  # elements on each side


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _guarded(T, d, dtype):
    buf = torch.full((GUARD * 2 + T * d,), 12345.0, device=dev(), dtype=dtype)
    return buf, buf[GUARD:GUARD + T * d].view(T, d)


def _guards_intact(buf):
    ref = torch.full((GUARD,), 12345.0, device=dev(), dtype=buf.dtype)
    return torch.equal(buf[:GUARD], ref) and torch.equal(buf[-GUARD:], ref)


@pytest.mark.parametrize("T,d", [(1, 896), (9, 1024), (101, 640), (13, 100)])
def test_full_read_stays_in_bounds(T, d):
    g = inputs.generator(20, dev())
    V = inputs.history(5, T, d, "bf16", g, dev())
    buf, out = _guarded(T, d, torch.bfloat16)
    ar.attnres_full_fwd(V, 5, inputs.queries(1, d, 0.1, g, dev())[0], torch.ones(d, device=dev()), 1e-6, out)
    torch.cuda.synchronize()
    assert _guards_intact(buf)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("T,d,S,n", [(5, 1024, 8, 8), (33, 2048, 6, 4), (3, 512, 3, 9)])
def test_stage1_stays_in_bounds(T, d, S, n):
    g = inputs.generator(21, dev())
    Src = inputs.history(n, T, d, "bf16", g, dev())
    bufs = [_guarded(T, d, torch.bfloat16) for _ in range(S)]
    lbuf, lse = _guarded(S, T, torch.float32)
    ar.attnres_block_stage1(Src, n, inputs.queries(S, d, 0.05, g, dev()), torch.ones(S, d, device=dev()),
                            1e-6, [o for _, o in bufs], lse.reshape(S, T))
    torch.cuda.synchronize()
    assert all(_guards_intact(b) for b, _ in bufs)
    assert _guards_intact(lbuf)


@pytest.mark.parametrize("T,d", [(3, 1024), (17, 2048), (5, 3)])
def test_merge_and_accumulate_stay_in_bounds(T, d):
    g = inputs.generator(22, dev())
    O = inputs.randn((T, d), "bf16", g, dev())
    lse = torch.zeros(T, device=dev())
    pbuf, P = _guarded(T, d, torch.float32)
    P.normal_()
    f = inputs.randn((T, d), "bf16", g, dev())
    obuf, out = _guarded(T, d, torch.bfloat16)
    ar.attnres_block_merge(O, lse, P, f, False, torch.ones(d, device=dev()), torch.ones(d, device=dev()),
                           1e-6, out)
    sbuf, summ = _guarded(T, d, torch.bfloat16)
    ar.attnres_block_summary_accumulate(P, f, False, summ)
    torch.cuda.synchronize()
    assert _guards_intact(pbuf) and _guards_intact(obuf) and _guards_intact(sbuf)


def test_device_status_clean_after_work():
    assert ar.attnres_device_status() == 0


def test_status_error_raised_from_binding():
    g = inputs.generator(23, dev())
    V = inputs.history(2, 4, 128, "bf16", g, dev())
    out = torch.empty(4, 128, device=dev(), dtype=torch.bfloat16)
    with pytest.raises(ar.AttnResError) as ei:
        ar.attnres_full_fwd(V, 0, torch.ones(128, device=dev()), torch.ones(128, device=dev()), 1e-6, out)
    assert ei.value.status == 1


def test_bounded_wait_runs_out_and_reports_timeout():
    """A device wait that nothing satisfies gives up, is reported as
    ATTNRES_ERR_TIMEOUT, and leaves the context usable (no GPU fault)."""
    assert ar.attnres_device_status() == 0
    ar.attnres_selftest_wait_timeout()
    assert ar.attnres_device_status() == 4          # ATTNRES_ERR_TIMEOUT
    assert ar.attnres_device_status() == 0          # the record was cleared
    g = inputs.generator(24, dev())
    V = inputs.history(3, 16, 256, "bf16", g, dev())
    out = torch.empty(16, 256, device=dev(), dtype=torch.bfloat16)
    ar.attnres_full_fwd(V, 3, torch.zeros(256, device=dev()), torch.ones(256, device=dev()), 1e-6, out)
    assert torch.allclose(out.float(), V.float().mean(0), rtol=1e-2, atol=1e-2)
    assert ar.attnres_device_status() == 0
