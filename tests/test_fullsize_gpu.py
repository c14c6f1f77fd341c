"""Full-size GPU parity on the benchmark's workloads, launched as the benchmark
launches them, against the oracle: every (sequence, KV head) unit's codes,
scales and window compared bit for bit (as digests of their bytes), and
attention compared within |d| <= 1e-3 + 1e-2 |ref| on many units and steps.

- Llama-3-8B decode cache (batch 32, ~8192 tokens, 4-bit, R 128, G 32):
  4 of the 32 layers (each layer is one cache launched the same way); all
  32 x 8 units of each; attention on 16 (layer, sequence) pairs over 3
  consecutive steps, the second of which flushes a group in every unit, and
  the persistent-warp kernel (kernel choice 4) on the last of them.
- Long video (432000 tokens as 30 appends of 14400, R 256, G 128, 4-bit):
  all 8 units; attention after every 8th of the 64 decode steps.
- 8-bit ragged batch (lengths drawn in [1024, 131072], G 64, Key spikes):
  all 8 units of every sequence; attention for all of them.

The oracle side runs per unit in spawned worker processes
(``tests/oracle_pool.py``).
"""

import numpy as np
import pytest

from kvq_inputs import gen
from oracle_pool import pool, unit_digest, unit_task

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-3, 1e-2


@pytest.fixture(scope="module")
def torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def kvq(torch):
    import quantized_kv_cache_02_gb300 as kvq
    kvq.load_library()
    return kvq


@pytest.fixture(scope="module")
def workers():
    p = pool()
    yield p
    p.close()
    p.join()


def close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, what
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    excess = np.abs(got - ref) - (ATOL + RTOL * np.abs(ref))
    w = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, f"{what}: |d| {abs(got - ref)[w]:.3e} at {w} (ref {ref[w]:.4e})"


def gpu_digest(cache, b, h):
    u = cache.export_unit(b, h)
    return unit_digest(u["k_codes"], u["v_codes"], u["k_scales"], u["v_scales"], u["window_k"], u["window_v"])


def task(spec, layer, b, h, R, G, qmax, chunks, attend_after=(), attend_steps=()):
    return dict(seed=spec.seed, n_kv_heads=spec.n_kv_heads, n_q_heads=spec.n_q_heads, head_dim=spec.head_dim,
                spikes=spec.spikes, layer=layer, seq=b, head=h, R=R, G=G, qmax=qmax, chunks=list(chunks),
                attend_after=list(attend_after), attend_steps=list(attend_steps))


def test_full_size_llama_batch32_four_layers(kvq, torch, workers):
    from kvq_inputs.device import DeviceInputs
    spec = gen.InputSpec(seed=2, n_kv_heads=8, n_q_heads=32, head_dim=128)
    B, H, Hq, D, R, G, qmax = 32, 8, 32, 128, 128, 32, 7
    g = Hq // H
    # window after the prefill: 8222 - 8064 = 158 tokens; the second step's
    # append fills it to R + G = 160 and flushes a group in every unit
    T0, steps = 8222, 3
    layers, att_seqs = (0, 9, 21, 31), (0, 11, 22, 31)
    dev = DeviceInputs(spec)
    tasks, keys = [], []
    for layer in layers:
        for b in range(B):
            for h in range(H):
                att = b in att_seqs
                tasks.append(task(spec, layer, b, h, R, G, qmax, [T0] + [1] * steps,
                                  attend_after=range(1, steps + 1) if att else (),
                                  attend_steps=range(steps) if att else ()))
                keys.append((layer, b, h))
    pending = workers.map_async(unit_task, tasks, chunksize=8)
    got_digest, got_out, got_line = {}, {}, {}
    for layer in layers:
        cache = kvq.KVQCache(B, H, Hq, D, R, G, qmax, T0 + 8)
        K, V = dev.kv_block(layer, 0, B, 0, T0)
        cache.append(K, V, 0)
        del K, V
        outs = []
        for s in range(steps):
            K, V = dev.kv_block(layer, 0, B, T0 + s, 1)
            cache.append(K, V, 0)
            q = dev.q_block(layer, 0, B, s)
            outs.append(cache.decode_attention(q).cpu().numpy())
            # the persistent-warp kernel on the same cache, last step
            if s == steps - 1:
                got_line[layer] = cache.decode_attention(q, kernel=4).cpu().numpy()
            if s == 1:
                assert all(cache.seq_state(b)["window"] == R for b in range(B)), "step 1 flushes a group"
        for b in range(B):
            for h in range(H):
                got_digest[(layer, b, h)] = gpu_digest(cache, b, h)
        got_out[layer] = np.stack(outs)  # [steps, B, Hq, D]
        assert cache.device_status() == 0
        del cache
        torch.cuda.empty_cache()
    results = dict(zip(keys, pending.get(timeout=900)))
    bad = [k for k in keys if results[k][0] != got_digest[k]]
    assert not bad, f"{len(bad)} units differ from the oracle's codes/scales/window, first {bad[:4]}"
    for layer in layers:
        for b in att_seqs:
            ref = np.stack([np.concatenate([results[(layer, b, h)][1][s] for h in range(H)]) for s in range(steps)])
            close(got_out[layer][:, b], ref, f"layer {layer} seq {b}")
            close(got_line[layer][b], ref[-1], f"layer {layer} seq {b}, persistent-warp kernel")
    assert g == 4


def test_full_size_long_video(kvq, torch, workers):
    from kvq_inputs.device import DeviceInputs
    spec = gen.InputSpec(seed=4, n_kv_heads=8, n_q_heads=32, head_dim=128)
    H, Hq, D, R, G, qmax = 8, 32, 128, 256, 128, 7
    chunk, n_chunks, steps = 14400, 30, 64
    T = chunk * n_chunks
    checked = list(range(7, steps, 8))
    tasks = [task(spec, 0, 0, h, R, G, qmax, [chunk] * n_chunks + [1] * steps,
                  attend_after=[n_chunks + s for s in checked], attend_steps=checked) for h in range(H)]
    pending = workers.map_async(unit_task, tasks, chunksize=1)
    dev = DeviceInputs(spec)
    cache = kvq.KVQCache(1, H, Hq, D, R, G, qmax, T + steps)
    for c in range(n_chunks):
        K, V = dev.kv_block(0, 0, 1, c * chunk, chunk)
        cache.append(K, V, 0)
    outs = {}
    for s in range(steps):
        K, V = dev.kv_block(0, 0, 1, T + s, 1)
        cache.append(K, V, 0)
        if s in checked:
            outs[s] = cache.decode_attention(dev.q_block(0, 0, 1, s)).cpu().numpy()[0]
    digests = [gpu_digest(cache, 0, h) for h in range(H)]
    assert cache.device_status() == 0
    results = pending.get(timeout=900)
    for h in range(H):
        assert results[h][0] == digests[h], f"head {h}: codes/scales/window differ from the oracle"
    for k, s in enumerate(checked):
        ref = np.concatenate([results[h][1][k] for h in range(H)])
        close(outs[s], ref, f"step {s}")


def test_full_size_ragged_8bit(kvq, torch, workers):
    from kvq_inputs.device import DeviceInputs
    spec = gen.InputSpec(seed=3, n_kv_heads=8, n_q_heads=32, head_dim=128, spikes=True)
    B, H, Hq, D, R, G, qmax = 4, 8, 32, 128, 128, 64, 127
    lens = spec.lengths(B, 1024, 131072)
    tasks = [task(spec, 0, b, h, R, G, qmax, [lens[b]], attend_after=[0], attend_steps=[0])
             for b in range(B) for h in range(H)]
    pending = workers.map_async(unit_task, tasks, chunksize=1)
    dev = DeviceInputs(spec)
    cache = kvq.KVQCache(B, H, Hq, D, R, G, qmax, [n + 8 for n in lens])
    for b, n in enumerate(lens):
        K, V = dev.kv_block(0, b, 1, 0, n)
        cache.append(K, V, b)
        del K, V
    out = cache.decode_attention(dev.q_block(0, 0, B, 0)).cpu().numpy()
    digests = {(b, h): gpu_digest(cache, b, h) for b in range(B) for h in range(H)}
    assert cache.device_status() == 0
    results = dict(zip([(b, h) for b in range(B) for h in range(H)], pending.get(timeout=900)))
    bad = [k for k in digests if results[k][0] != digests[k]]
    assert not bad, f"units differ from the oracle: {bad}"
    for b in range(B):
        ref = np.concatenate([results[(b, h)][1][0] for h in range(H)])
        close(out[b], ref, f"seq {b} (T={lens[b]})")
