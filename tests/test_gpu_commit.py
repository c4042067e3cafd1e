"""GPU parity: eagle_kv_commit against the oracle's commit (exact bytes).

Also: a request whose commit would pass the cache capacity is left untouched and
flagged, a path node outside the tree is flagged, and feature rows (including a
width that is not a multiple of 16 bytes) follow the path.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_tree_gb300 import binding as B
from eagle_speculative_decoding_tree_gb300 import synth

pytestmark = pytest.mark.gpu


def _bf16(g, shape):
    return synth.bf16_bits(synth.normal_row(g, shape, 1.0))


def _run(kc, vc, tk, tv, n_acc, path, seq_len, max_seq, feat=None, tfeat=None, feat_dtype=B.EAGLE_F32):
    L, Bn, H, P, D = kc.shape
    R = tk.shape[3]
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    kcs = [to_t(kc[l].copy()) for l in range(L)]
    vcs = [to_t(vc[l].copy()) for l in range(L)]
    tks = [to_t(tk[l].copy()) for l in range(L)]
    tvs = [to_t(tv[l].copy()) for l in range(L)]
    layers = B.LayerPointers(kcs, vcs, tks, tvs)
    fd = 0 if feat is None else feat.shape[-1]
    desc = B.CommitDesc(L, Bn, H, D, R, max_seq, path.shape[1] - 1, B.EAGLE_BF16, fd, feat_dtype)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    sl = i32(seq_len)
    pos = torch.zeros(path.shape, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if feat is not None:
        conv = (lambda a: torch.from_numpy(a.copy()).cuda()) if feat_dtype == B.EAGLE_F32 else to_t
        fc, tf = conv(feat), conv(tfeat)
    else:
        fc = tf = None
    B.eagle_kv_commit(desc, layers, i32(n_acc), i32(path), sl, pos, fc, tf, status)
    torch.cuda.synchronize()
    back = lambda ts: np.stack([t.view(torch.int16).cpu().numpy().view(np.uint16) for t in ts])
    fout = None
    if fc is not None:
        fout = fc.cpu().numpy() if feat_dtype == B.EAGLE_F32 else fc.view(torch.int16).cpu().numpy().view(np.uint16)
    return back(kcs), back(vcs), sl.cpu().numpy(), pos.cpu().numpy(), int(status.cpu()[0]), fout


def test_commit_matches_oracle_bytes():
    g = synth.rng(0, 6100)
    L, Bn, H, P, R, D, maxd = 4, 3, 8, 96, 61, 128, 7
    kc, vc = _bf16(g, (L, Bn, H, P, D)), _bf16(g, (L, Bn, H, P, D))
    tk, tv = _bf16(g, (L, Bn, H, R, D)), _bf16(g, (L, Bn, H, R, D))
    feat, tfeat = synth.normal_row(g, (Bn, P, 96), 1.0), synth.normal_row(g, (Bn, R, 96), 1.0)
    seq_len = np.array([40, 0, 88], np.int32)
    n_acc = np.array([7, 0, 3], np.int32)
    path = np.full((Bn, maxd + 1), -1, np.int32)
    path[0] = [0, 3, 9, 20, 33, 41, 50, 60]
    path[1, 0] = 0
    path[2, :4] = [0, 1, 2, 5]
    gk, gv, gsl, gpos, st, gf = _run(kc, vc, tk, tv, n_acc, path, seq_len, P, feat, tfeat)
    rk, rv, rf = kc.copy(), vc.copy(), feat.copy()
    rsl, rpos = oracle.kv_commit(rk, rv, tk, tv, n_acc, path, seq_len, rf, tfeat)
    assert gk.tobytes() == rk.tobytes() and gv.tobytes() == rv.tobytes()
    assert gf.tobytes() == rf.tobytes()
    assert np.array_equal(gsl, rsl) and np.array_equal(gpos, rpos)
    assert st == 0


def test_commit_cache_full_is_flagged_and_untouched():
    g = synth.rng(0, 6200)
    L, Bn, H, P, R, D = 2, 2, 2, 64, 11, 64
    kc, vc = _bf16(g, (L, Bn, H, P, D)), _bf16(g, (L, Bn, H, P, D))
    tk, tv = _bf16(g, (L, Bn, H, R, D)), _bf16(g, (L, Bn, H, R, D))
    seq_len = np.array([60, 10], np.int32)   # request 0: 60 + 4 + 1 > 64
    n_acc = np.array([4, 2], np.int32)
    path = np.array([[0, 1, 5, 9, 10], [0, 2, 7, -1, -1]], np.int32)
    gk, gv, gsl, gpos, st, _ = _run(kc, vc, tk, tv, n_acc, path, seq_len, P)
    assert st & B.EAGLE_STATUS_CACHE_FULL
    assert gsl.tolist() == [60, 13]
    assert gk[:, 0].tobytes() == kc[:, 0].tobytes()
    assert gpos[0].tolist() == [-1] * 5 and gpos[1].tolist() == [10, 11, 12, -1, -1]
    for m, node in enumerate([0, 2, 7]):
        assert gk[:, 1, :, 10 + m].tobytes() == tk[:, 1, :, node].tobytes()


def test_commit_bad_path_node_is_flagged():
    g = synth.rng(0, 6300)
    L, Bn, H, P, R, D = 1, 1, 1, 32, 5, 64
    kc, vc = _bf16(g, (L, Bn, H, P, D)), _bf16(g, (L, Bn, H, P, D))
    tk, tv = _bf16(g, (L, Bn, H, R, D)), _bf16(g, (L, Bn, H, R, D))
    _, _, _, _, st, _ = _run(kc, vc, tk, tv, np.array([1], np.int32), np.array([[0, 9]], np.int32),
                             np.array([3], np.int32), P)
    assert st & B.EAGLE_STATUS_BAD_TREE


def test_commit_feature_rows_bf16_odd_width():
    g = synth.rng(0, 6400)
    L, Bn, H, P, R, D = 1, 2, 2, 40, 11, 64
    kc, vc = _bf16(g, (L, Bn, H, P, D)), _bf16(g, (L, Bn, H, P, D))
    tk, tv = _bf16(g, (L, Bn, H, R, D)), _bf16(g, (L, Bn, H, R, D))
    feat, tfeat = _bf16(g, (Bn, P, 100)), _bf16(g, (Bn, R, 100))  # 200-byte rows
    n_acc = np.array([2, 1], np.int32)
    path = np.array([[0, 2, 6], [0, 4, -1]], np.int32)
    seq_len = np.array([5, 30], np.int32)
    _, _, _, _, st, gf = _run(kc, vc, tk, tv, n_acc, path, seq_len, P, feat, tfeat, B.EAGLE_BF16)
    rf = feat.copy()
    rk, rv = kc.copy(), vc.copy()
    oracle.kv_commit(rk, rv, tk, tv, n_acc, path, seq_len, rf, tfeat)
    assert st == 0 and gf.tobytes() == rf.tobytes()
