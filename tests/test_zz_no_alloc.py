"""The allocation-free decode entry point (GPU).

fa_decode_noalloc is for callers that must not allocate device memory where
they run (allocator callbacks, runtimes that own all device memory, plugins
handed only their buffers); it keeps its split-K partials in a fixed array
inside the library.  This file checks, through the C ABI, that two calls in a
row give what fa_decode gives with a caller workspace on the same inputs --
so the array's leftover contents from the first call cannot leak into the
second -- and that a problem too large for the array is refused.

It sits last in collection order and works both alone and after the others.
"""

import numpy as np
import pytest
import torch

from attention_forward_16_gb300 import binding as fb
from attention_forward_16_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

TOL = 1e-5  # the decode tests' bound on fp32-compared outputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_16_gb300.build import build
    build()
    fb.load()


def _inputs(seed, B=2, H=4, Nq=2, Nk=3000, D=128, dtype="bf16"):
    q, _, _ = make_qkv(B, H, Nq, D, dtype, seed=seed, n_k=1)
    _, k, v = make_qkv(B, H, 1, D, dtype, seed=seed + 1, n_k=Nk)
    return q.cuda(), k.cuda(), v.cuda()


def _split_count(q, k):
    """The split count fa_decode would choose for this shape.  Both entry
    points are then given it explicitly: with the same splits they do the
    same arithmetic in the same order, so the comparison is exact whatever
    rule either one would use to choose its own count."""
    B, H, Nq, D = q.shape
    ns, wb = fb.fa_decode_plan(B, H, Nq, k.shape[2], D, 0)
    assert ns > 1 and wb > 0, "the shape must need partials for the comparison to mean anything"
    return ns


def _with_workspace(q, k, v, mk, ns, stream):
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    ns_out, wb = fb.fa_decode_plan(B, H, Nq, Nk, D, ns)
    assert ns_out == ns
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    rc = fb.fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk, D,
                      0.09, mk, -1, -1, fb.FA_BF16, ns, ws.data_ptr(), wb, stream)
    assert rc == fb.FA_OK
    return o, lse


def _no_alloc(q, k, v, mk, ns, stream):
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    rc = fb.fa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Nq, Nk,
                              D, 0.09, mk, -1, -1, fb.FA_BF16, ns, stream)
    assert rc == fb.FA_OK, fb.load().fa_strerror(rc)
    return o, lse


def test_no_alloc_matches_workspace_entry_point_twice_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    first = _inputs(seed=300)
    second = _inputs(seed=400)
    results = []
    for (q, k, v), mk in ((first, fb.FA_MASK_CAUSAL), (second, fb.FA_MASK_NONE)):
        ns = _split_count(q, k)
        results.append((_no_alloc(q, k, v, mk, ns, stream), _with_workspace(q, k, v, mk, ns, stream)))
    torch.cuda.synchronize()
    assert fb.fa_device_status(stream) == fb.FA_OK
    for (o_na, l_na), (o_ws, l_ws) in results:
        assert np.abs(o_na.float().cpu().numpy() - o_ws.float().cpu().numpy()).max() <= TOL
        assert np.abs(l_na.cpu().numpy() - l_ws.cpu().numpy()).max() <= TOL
    # the two calls computed different problems: the second did not reuse the first's partials
    assert not torch.equal(results[0][0][0], results[1][0][0])


def test_no_alloc_refuses_problems_beyond_its_scratch():
    cap = fb.fa_decode_noalloc_scratch_bytes()
    assert cap == 16 << 20
    B, H, Nq, Nk, D, ns = 64, 32, 16, 4096, 128, 16
    _, need = fb.fa_decode_plan(B, H, Nq, Nk, D, ns)
    assert need > cap
    buf = torch.empty(64, dtype=torch.bfloat16, device="cuda")   # never read: the call returns before launching
    p = buf.data_ptr()
    rc = fb.fa_decode_noalloc(p, p, p, p, None, B, H, Nq, Nk, D, 0.09, fb.FA_MASK_NONE, -1, -1, fb.FA_BF16, ns,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == fb.FA_ERR_SCRATCH
    assert b"scratch" in fb.load().fa_strerror(rc)
