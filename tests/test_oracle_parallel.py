"""The parallel oracle driver of the GPU parity tests (experts in worker
processes) gives exactly the serial oracle's forward, and the tile-covering
token set covers every expert's tiles."""

import numpy as np

import synthetic
from oracle import moe as omoe
from tests.parity import oracle_forward, oracle_forward_parallel, oracle_route, tile_covering_tokens


def test_parallel_oracle_equals_serial():
    wl = synthetic.make_workload("c0_tiny")
    for tokens in (np.arange(wl.T), np.array([0, 3, 7, 15])):
        ref = oracle_forward(wl, tokens)
        out, ids, h_gs = oracle_forward_parallel(wl, tokens)
        assert np.array_equal(ids, ref.ids)
        assert np.array_equal(out.view(np.uint32), ref.out.view(np.uint32))
        assert h_gs.keys() == ref.h_gs.keys()
        assert all(h_gs[k] == ref.h_gs[k] for k in h_gs)


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
