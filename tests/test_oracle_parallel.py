"""The parallel oracle driver of the GPU parity tests (experts in worker
processes) gives exactly the serial oracle's forward; fed the oracle's own
intermediate as the "GPU" one it reports no flipped block and the same
output; a planted flip is counted; and the tile-covering token set covers
every expert's tiles."""

import numpy as np

import synthetic
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.parity import oracle_forward, oracle_forward_parallel, oracle_route, tile_covering_tokens


def _oracle_intermediate(wl):
    """The oracle's requantized intermediate of every (token, slot), indexed
    by token * K + slot: packed codes, block scales, global scales."""
    x = omoe.as_f32(wl.x)
    K, I = wl.shape.K, wl.shape.I
    _, ids, _ = oracle_route(wl)
    xc, xs, xg = onv.quantize_rows(x)
    q13 = omoe.quantize_weights(omoe.as_f32(wl.w13))
    q2 = omoe.quantize_weights(omoe.as_f32(wl.w2))
    codes = np.zeros((wl.T * K, I // 2), np.uint8)
    sf = np.zeros((wl.T * K, I // 16), np.uint8)
    gs = np.zeros(wl.T * K, np.float32)
    for e in np.unique(ids):
        t, j = np.nonzero(ids == e)
        r = omoe.expert_rows(xc[t], xs[t], xg[t], q13, q2, int(e))
        src = t * K + j
        codes[src], sf[src], gs[src] = onv.pack_e2m1(r["h_codes"]), r["h_sf"], r["h_gs"]
    return codes, sf, gs


def test_parallel_oracle_equals_serial():
    wl = synthetic.make_workload("c0_tiny")
    for tokens in (np.arange(wl.T), np.array([0, 3, 7, 15])):
        ref = oracle_forward(wl, tokens)
        res = oracle_forward_parallel(wl, tokens)
        assert np.array_equal(res.ids, ref.ids)
        assert np.array_equal(res.out.view(np.uint32), ref.out.view(np.uint32))
        assert res.h_gs.keys() == ref.h_gs.keys()
        assert all(res.h_gs[k] == ref.h_gs[k] for k in res.h_gs)


def test_downstream_of_a_given_intermediate():
    wl = synthetic.make_workload("c0_tiny")
    h = _oracle_intermediate(wl)
    tokens = np.array([1, 4, 9, 15])
    res = oracle_forward_parallel(wl, tokens, h_gpu=h)
    assert res.flipped_blocks == 0 and not res.flipped.any()
    assert res.blocks == len(tokens) * wl.shape.K * wl.shape.I // 16
    assert np.array_equal(res.out_gpu_h.view(np.uint32), res.out.view(np.uint32))
    assert np.array_equal(res.h_gs_gpu.view(np.uint32), res.h_gs_ref.view(np.uint32))
    # a planted flip: one code of token 9's slot-1 row moves to its neighbour
    codes = h[0].copy()
    src = 9 * wl.shape.K + 1
    codes[src, 3] ^= 0x01
    res2 = oracle_forward_parallel(wl, tokens, h_gpu=(codes, h[1], h[2]))
    assert res2.flipped_blocks == 1
    assert res2.flipped[2, 1] and res2.flipped.sum() == 1
    assert not np.array_equal(res2.out_gpu_h[2], res2.out[2])
    assert np.array_equal(res2.out_gpu_h[[0, 1, 3]], res2.out[[0, 1, 3]])


def test_tile_covering_tokens():
    wl = synthetic.make_workload("c0_tiny")
    _, ids, _ = oracle_route(wl)
    E, K = wl.shape.E, wl.shape.K
    tiles = 3  # rows per tile, so that experts span several tiles with a ragged last one
    toks = set(tile_covering_tokens(ids, E, tiles).tolist())
    off, src, _ = omoe.permute(ids, E)
    for e in range(E):
        n = int(off[e + 1] - off[e])
        for r0 in range(0, n, tiles):
            rows = range(r0, min(r0 + tiles, n))
            assert any(int(src[off[e] + r]) // K in toks for r in rows), (e, r0)
            assert int(src[off[e] + rows[-1]]) // K in toks
