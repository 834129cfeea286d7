"""Calls chained inside CUDA graphs and replayed.

The pages report a bug where a compiler moved one call's read past the next
call's write to a shared buffer, and conclude that every kernel test should
chain calls under CUDA graphs ("What Broke in Production").  Here a graph
captures write -> attention -> write -> attention on one ring (ring state is
device-resident, so every replay advances the ring), and another graph holds
a delta rotation; replays are checked against the oracle after each step.
"""
import numpy as np
import pytest
import torch

import ring_kv_cache_gb300 as kv
from oracle import Ring, TO_OLDEST
from oracle.attention import attention_exact
from workloads import TINY, tiny_session

from _ringcheck import MAX_ABS, MEAN_ABS, assert_ring_equal, attn_errors, dev, f, make_pair

pytestmark = pytest.mark.gpu


def test_graph_chain_replays_match_oracle():
    frames = tiny_session(frames=14)
    ring, orc = make_pair(TINY, Ring)
    ring.calibrate(dev(frames[0][1]), dev(frames[0][2]))
    orc.calibrate(f(frames[0][1]), f(frames[0][2]))
    ring.write(dev(frames[0][1]), dev(frames[0][2]))
    orc.write(f(frames[0][1]), f(frames[0][2]))
    torch.cuda.synchronize()

    kin = [torch.empty((12, 2, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    vin = [torch.empty_like(kin[0]) for _ in range(2)]
    qin = [torch.empty_like(kin[0]) for _ in range(2)]
    outs = [torch.empty((12, 2, 64), dtype=torch.float32, device="cuda") for _ in range(2)]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for j in range(2):
            ring.write(kin[j], vin[j])
            ring.attention(qin[j], out=outs[j])
    g_reset = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_reset, stream=s):
        ring.delta_rotate(kv.TO_OLDEST)

    fi = 1
    for rep in range(6):
        if rep == 4:
            g_reset.replay()
            orc.delta_rotate(TO_OLDEST)
        for j in range(2):
            qf, kf, vf = frames[fi + j]
            kin[j].copy_(dev(kf))
            vin[j].copy_(dev(vf))
            qin[j].copy_(dev(qf))
        g.replay()
        torch.cuda.synchronize()
        for j in range(2):
            qf, kf, vf = frames[fi + j]
            orc.write(f(kf), f(vf))
            want = attention_exact(orc, f(qf))
            mx, mn = attn_errors(outs[j].cpu().numpy(), want)
            assert mx <= MAX_ABS and mn <= MEAN_ABS, (rep, j, mx, mn)
        assert_ring_equal(ring, orc, f"replay {rep}")
        fi = (fi + 2) % 12 + 1
