"""GPU: eagle_accept_noalloc (scratch in the library's fixed device buffer) against
eagle_accept (caller workspace) on the same inputs, two calls in a row; and the
host-side rejection of a descriptor whose scratch exceeds the buffer.

The two entry points run the same kernels, so their outputs (accepted lengths,
paths, emitted tokens, near-tie flags, status words: all integers) must agree
exactly.  The file name sorts last so that the test also runs after the rest of
the GPU suite; it needs no state from it.
"""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import step, synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20  # EAGLE_ACCEPT_NOALLOC_SCRATCH_BYTES


def _outputs(acc):
    return {k: getattr(acc, k).cpu().numpy().copy() for k in ("n_acc", "path", "out_tok", "near_tie", "status")}


@pytest.mark.parametrize("name", ["llama8b", "vicuna7b"])
def test_noalloc_matches_workspace_entry_point(name):
    w = synth.WORKLOADS[name]
    vs = step.VerifyStep(w, batch=2, layers=1)
    assert B.workspace_size(B.EAGLE_WS_ACCEPT, vs.acc_desc) <= SCRATCH_BYTES
    vs.accept()
    torch.cuda.synchronize()
    ref = _outputs(vs.acc)
    for call in range(2):
        got = B.AcceptBuffers.allocate(vs.B, vs.max_depth, torch.device("cuda"))
        B.eagle_accept_noalloc(vs.acc_desc, vs.target, vs.draft, vs.tokens, vs.parent, vs.u_accept, vs.u_final, got)
        torch.cuda.synchronize()
        out = _outputs(got)
        for k in ref:
            assert np.array_equal(out[k], ref[k]), (call, k, out[k], ref[k])


def test_noalloc_rejects_scratch_beyond_the_buffer():
    # 128 requests x 61 rows at vocab 128256 need 128 * 61 * 768 bytes > 4 MiB; the
    # call is refused on the host, before any launch.
    d = B.AcceptDesc(128, 61, 128256, 1.0, B.EAGLE_PROPOSAL_DELTA, B.EAGLE_BF16, 7)
    assert B.workspace_size(B.EAGLE_WS_ACCEPT, d) > SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = t.data_ptr()
    o = B.AcceptOut(p, p, p, p, p)
    rc = B.load().eagle_accept_noalloc(d, p, None, p, p, p, p, o, None)
    assert rc == B.EAGLE_ERR_WORKSPACE
