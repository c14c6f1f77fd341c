"""Oracle work for the full-size GPU parity tests, one (layer, sequence, KV
head) unit per task, run in spawned worker processes.

Test infrastructure: it calls only the oracle (``oracle.kvq_oracle``) and the
seeded input generator.  A unit's quantizer and attention depend on no other
KV head (Key scales per channel and Value scales per token are taken per
head; query head h reads KV head h // g), so each task builds a one-head
``GroupedSequence`` and its result is exactly that head's part of the full
oracle.  Codes, scales and the window are returned as a SHA-256 digest of
their bytes (compared with the same digest of what the GPU cache exports);
attention outputs as float64 arrays.
"""

from __future__ import annotations

import hashlib
import multiprocessing as mp
import os

import numpy as np


def unit_digest(k_codes, v_codes, k_scales, v_scales, window_k, window_v) -> str:
    """Digest of one unit's held state: int8 codes, fp32 scales, fp32 window,
    in this order, each as C-contiguous bytes."""
    h = hashlib.sha256()
    for a, dt in ((k_codes, np.int8), (v_codes, np.int8), (k_scales, np.float32), (v_scales, np.float32),
                  (window_k, np.float32), (window_v, np.float32)):
        h.update(np.ascontiguousarray(a, dtype=dt).tobytes())
    return h.hexdigest()


def unit_task(args: dict):
    """One (layer, seq, head) unit.  ``args``: seed, n_kv_heads, n_q_heads,
    head_dim, spikes, layer, seq, head, R, G, qmax, chunks (the appends, in
    tokens: a prefill split as the GPU side appends it, then single tokens),
    attend_after (indices into ``chunks`` after which to attend, with the
    query of step ``attend_steps[k]``).  Returns (digest, [outputs])."""
    from kvq_inputs import gen
    from oracle import kvq_oracle as O
    spec = gen.InputSpec(seed=args["seed"], n_kv_heads=args["n_kv_heads"], n_q_heads=args["n_q_heads"],
                         head_dim=args["head_dim"], spikes=args.get("spikes", False))
    layer, b, h = args["layer"], args["seq"], args["head"]
    g = args["n_q_heads"] // args["n_kv_heads"]
    seq = O.GroupedSequence(1, args["head_dim"], args["R"], args["G"], args["qmax"])
    outs = []
    attend = dict(zip(args.get("attend_after", []), args.get("attend_steps", [])))
    t = 0
    for i, n in enumerate(args["chunks"]):
        k, v = spec.kv_block(layer, [b], t, n, heads=[h])
        seq.append(k[0], v[0])
        t += n
        if i in attend:
            q = spec.q_block(layer, [b], attend[i])[0, h * g:(h + 1) * g]
            outs.append(seq.attend(q))
    wk, wv = seq.window_kv()
    digest = unit_digest(seq.key_codes()[0], seq.value_codes()[0], seq.key_scales()[0], seq.value_scales()[0],
                         wk[0], wv[0])
    return digest, outs


def pool(processes: int | None = None):
    """A spawn-context pool (safe to start after CUDA is initialised)."""
    n = processes or min(16, os.cpu_count() or 4)
    return mp.get_context("spawn").Pool(n)
