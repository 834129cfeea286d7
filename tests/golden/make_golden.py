"""Writes tests/golden/tiny_session_oracle.txt from the oracle alone.

Runs the tiny workload (2 heads of 64, 48 slots, 12 tokens per frame, 10
frames, positions frame*12 + token, scales from frame 0, one delta rotation
to the oldest slot before frame 7) through ``oracle.Ring`` and records
SHA-256 digests of the final cache bytes, positions and scales, plus a few
attention values.  The stored file pins the oracle across machines (x86 and
Arm libm, numpy builds); it never holds a value produced by the CUDA path.

Usage: python tests/golden/make_golden.py
"""
import hashlib
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import Ring, TO_OLDEST  # noqa: E402
from oracle.attention import attention_exact  # noqa: E402
from workloads import TINY, f32_from_bf16, tiny_session  # noqa: E402


def run_tiny():
    frames = tiny_session()
    r = Ring(TINY.heads, TINY.head_dim, TINY.capacity, TINY.max_position, TINY.rope_base)
    r.calibrate(f32_from_bf16(frames[0][1]), f32_from_bf16(frames[0][2]))
    outs = []
    for f, (q, k, v) in enumerate(frames):
        if f == 7:
            r.delta_rotate(TO_OLDEST)
        r.write(f32_from_bf16(k), f32_from_bf16(v))
        outs.append(attention_exact(r, f32_from_bf16(q)))
    return r, outs


def digest(a) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def records():
    r, outs = run_tiny()
    rec = {
        "k_codes_sha256": digest(r.K),
        "v_codes_sha256": digest(r.V),
        "slot_pos_sha256": digest(r.slot_pos.astype(np.int64)),
        "scale_k_hex": " ".join(f"{x:08x}" for x in r.scale_k.view(np.uint32)),
        "scale_v_hex": " ".join(f"{x:08x}" for x in r.scale_v.view(np.uint32)),
        "state": f"head={r.head} n_valid={r.n_valid} total={r.total} next_pos={r.next_pos}",
        "attn_last_0_0_0_to_3": " ".join(f"{float(x):.10e}" for x in outs[-1][0, 0, :4]),
    }
    return rec


if __name__ == "__main__":
    rec = records()
    path = os.path.join(HERE, "tiny_session_oracle.txt")
    with open(path, "w") as f:
        f.write("# Oracle state after the tiny workload (see make_golden.py); written by the oracle only.\n")
        for k, v in rec.items():
            f.write(f"{k}: {v}\n")
    print(open(path).read())
