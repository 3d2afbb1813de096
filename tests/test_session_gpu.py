"""The host-buffer session (fa_session_*): one forward + backward step on CPU
tensors, pipelined over chunks of heads, must give exactly the outputs of
fa_forward + fa_backward on the whole batch on the device (heads are independent,
and each output element is computed by one thread block in a fixed order)."""
import pytest
import torch

import exact_io_aware_27_gb300 as fa
from exact_io_aware_27_gb300 import inputs as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fa.build()


def _device_reference(Q, K, V, dO, causal, scale):
    q, k, v, do = (t.cuda() for t in (Q, K, V, dO))
    O, L = fa.fa_forward(q, k, v, causal, scale)
    dQ, dK, dV = fa.fa_backward(q, k, v, O, L, do, causal, scale)
    torch.cuda.synchronize()
    return [t.cpu() for t in (O, L, dQ, dK, dV)]


@pytest.mark.parametrize("B,H,n,m,d,causal,chunk", [
    (2, 3, 300, 257, 64, True, 1),
    (2, 3, 300, 257, 64, True, 4),     # 6 heads in chunks of 4 and 2
    (1, 4, 128, 128, 128, False, 4),   # one chunk
    (1, 8, 513, 513, 128, True, 3),    # more chunks than buffer sets
    (1, 2, 100, 100, 32, False, 1),    # a head dimension below 64
])
def test_session_matches_device_path(B, H, n, m, d, causal, chunk):
    Q, K, V, dO = wl.attention_inputs(B, H, n, m, d, seed=8300 + n + d)
    ref = _device_reference(Q, K, V, dO, causal, None)
    sess = fa.Session(B, H, n, m, d, chunk)
    try:
        pinned = [t.pin_memory() for t in (Q, K, V, dO)]
        got = sess.step(*pinned, causal=causal)
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), got, ref):
            assert torch.equal(a, b), name
        # pageable host memory gives the same results, and a session runs many steps
        got2 = sess.step(Q, K, V, dO, causal=causal)
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), got2, ref):
            assert torch.equal(a, b), name
    finally:
        sess.close()
    assert fa.fa_get_device_status() == 0


def test_session_rejects_device_or_misshaped_inputs():
    Q, K, V, dO = wl.attention_inputs(1, 2, 64, 64, 64, seed=8400)
    sess = fa.Session(1, 2, 64, 64, 64, 1)
    try:
        with pytest.raises(ValueError):
            sess.step(Q.cuda(), K, V, dO)
        with pytest.raises(ValueError):
            sess.step(Q[:, :1].contiguous(), K, V, dO)
    finally:
        sess.close()


@pytest.mark.parametrize("B,H,n,m,d,causal,chunk", [
    (2, 3, 300, 257, 64, True, 4),     # 2 chunks a step: buffer sets reused across steps
    (1, 8, 513, 513, 128, True, 3),    # 4 chunks a step
    (1, 1, 200, 77, 64, False, 1),     # 1 chunk a step
])
def test_submitted_steps_overlap_and_match(B, H, n, m, d, causal, chunk):
    """Three steps submitted back to back, each on its own inputs and into its own
    output buffers, then one sync: each step's outputs equal the device path's for
    its inputs, so the pipeline that continues across steps keeps every chunk's
    buffer set apart from its neighbours' and from the previous step's."""
    batches = [wl.attention_inputs(B, H, n, m, d, seed=8500 + 10 * i + n) for i in range(3)]
    refs = [_device_reference(*b, causal, None) for b in batches]
    sess = fa.Session(B, H, n, m, d, chunk)
    try:
        outs = []
        for b in batches:
            pinned = [t.pin_memory() for t in b]
            outs.append((pinned, sess.submit(*pinned, causal=causal)))
        sess.sync()
        for i, ((_, got), ref) in enumerate(zip(outs, refs)):
            for name, a, r in zip(("O", "L", "dQ", "dK", "dV"), got, ref):
                assert torch.equal(a, r), f"step {i} {name}"
        # a blocking step after submitted ones continues the same pipeline
        got = sess.step(*[t.pin_memory() for t in batches[0]], causal=causal)
        for name, a, r in zip(("O", "L", "dQ", "dK", "dV"), got, refs[0]):
            assert torch.equal(a, r), name
    finally:
        sess.close()
    assert fa.fa_get_device_status() == 0
