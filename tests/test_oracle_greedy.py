"""Pin: greedy speculative decoding emits exactly the plain argmax decode.

The pages state that verification is lossless for greedy decoding as well (EAGLE
review, sections 3.3 and 4).  The target here is a synthetic LM whose rows are a
pure function of the token path, so plain argmax decoding is well defined and the
speculative loop (tree build, verify, accept, commit to the context) must
reproduce it token for token, whatever tree the draft proposes.
"""
import numpy as np
import pytest

import oracle
from eagle_speculative_decoding_tree_gb300 import synth
from spec_helpers import OracleDynamicBuilder, OracleStaticBuilder, drive_tree_build, node_hashes


def _argmax_decode(lm, h, n):
    out = []
    for _ in range(n):
        t = int(np.argmax(lm.target_row(h)))  # numpy's argmax takes the first maximum
        out.append(t)
        h = synth.child_hash(h, t)
    return out


def _speculative_decode(lm, h, root_tok, n, make_builder, depth):
    stream, steps, accepted = [], 0, []
    while len(stream) < n:
        bld = make_builder()
        tree = drive_tree_build(bld, lm, depth, np.array([root_tok], np.int32), [h], np.zeros(1, np.int32))
        hs = node_hashes(tree, [h])[0]
        tgt = synth.as_dtype_bytes(lm.rows(hs, "target")[None], lm.dtype)
        R = tree["tokens"].shape[1]
        res = oracle.accept(tgt, tree["tokens"], tree["parent"], np.zeros((1, R), np.float32),
                            np.zeros(1, np.float32), 0.0, oracle.DELTA, depth + 1)
        na = int(res["n_acc"][0])
        emitted = res["out_tok"][0, : na + 1].tolist()
        stream += emitted
        accepted.append(na)
        h = synth.child_hash(hs[int(res["path"][0, na])], emitted[-1])
        root_tok = emitted[-1]
        steps += 1
    return stream[:n], steps, accepted


@pytest.mark.parametrize("tree_kind", ["dynamic", "static_topk"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_speculative_equals_argmax_decoding(tree_kind, dtype):
    V, n = 40, 60
    # a strongly correlated draft so that several drafts get accepted per step
    lm = synth.HashLM(V, "normal", 3.0, 0.8, dtype)
    h0 = synth.root_hash(0, 1, 77)
    if tree_kind == "dynamic":
        mk, depth = (lambda: OracleDynamicBuilder(1, V, 4, 4, 12)), 4
    else:
        par = synth.static_parents(synth.TINY_STATIC_CHOICES)
        mk, depth = (lambda: OracleStaticBuilder(1, V, par, False, 0.0)), 3
    spec, steps, accepted = _speculative_decode(lm, h0, 5, n, mk, depth)
    assert spec == _argmax_decode(lm, h0, n)
    assert steps < n  # some drafts were accepted
    assert max(accepted) >= 2
