"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

For each workload (32K, ragged paged batch, 196K with drift, batch-64 GQA-5 with
9-bit values, 32K in the 1.5-bit configuration): the whole cache is encoded on the GPU (prefill plus the appended
token) and decoded with the library's default split count and launch shape.
The oracle then checks sampled (sequence, KV head) pairs one by one:
  - the codes of all N + 1 tokens: bit-exact except in-band ties (logged);
  - the attention rows of the pair, after the pair's rows of the pools are
    overwritten with the oracle's own codes and the same launch runs again,
    against the fp64 oracle over those codes (inputs flow from the oracle to
    the GPU, never back), within max-abs 2e-3 / mean-abs 2e-4;
  - when the pair's codes had no tie, the end-to-end rows of the first launch
    against the same oracle result.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import (GpuCache, check_outputs, compare_codes, oracle_attention, oracle_encode,
                    skip_end_to_end, stored_calib, write_tie_log)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_full_size_sampled_parity(cfg):
    w = W.WORKLOADS[cfg]
    cal = stored_calib(cfg)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    q = W.queries(w)
    got = gc.decode(q)
    assert gc.device_status() == 0
    assert np.isfinite(got).all()
    G = w.num_q_heads // w.num_kv_heads
    rng = np.random.default_rng(4000 + cfg)
    pairs = {(int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads)))
             for _ in range(1 if cfg in (3, 5) else 2)}
    pairs.add((w.batch - 1, w.num_kv_heads - 1))
    log, refs, tied = [], {}, {}
    for b, h in sorted(pairs):
        n = int(gc.lens[b]) + 1                      # cached tokens + the appended one
        r = oracle_encode(w, cal, b, 0, n, heads=[h])
        kc, vc = gc.codes(b, 0, n, heads=[h])
        ties = compare_codes(kc, r.kc, r.kx, cal.ck, w.k_sub, f"cfg{cfg}/k/b{b}h{h}", log)
        ties += compare_codes(vc, r.vc, r.vx, cal.cv, w.v_sub, f"cfg{cfg}/v/b{b}h{h}", log)
        tied[(b, h)] = ties
        refs[(b, h)] = oracle_attention(w, cal, q[b, h * G:(h + 1) * G], r.kc, r.vc, heads=[h])
        gc.write_codes(b, 0, r.kc, r.vc, heads=[h])
    write_tie_log(f"full_cfg{cfg}", log)
    again = gc.decode(q)
    assert gc.device_status() == 0
    for (b, h), ref in sorted(refs.items()):
        rows = slice(h * G, (h + 1) * G)
        check_outputs(again[b, rows], ref, f"cfg{cfg} b{b} kv-head {h}, oracle codes")
        if tied[(b, h)] == 0:
            check_outputs(got[b, rows], ref, f"cfg{cfg} b{b} kv-head {h}, end to end")
        else:
            skip_end_to_end(f"cfg{cfg} b{b} kv-head {h}", tied[(b, h)])


def test_full_size_codes_exhaustive_llama_32k():
    """Every code of the 32K workload (8 KV heads x 32769 tokens, K and V)
    against the oracle: bit-exact except in-band ties."""
    w = W.WORKLOADS[1]
    cal = stored_calib(1)
    gc = GpuCache(w, cal)
    gc.prefill()
    gc.append()
    assert gc.device_status() == 0
    n = int(gc.lens[0]) + 1
    log = []
    r = oracle_encode(w, cal, 0, 0, n)
    kc, vc = gc.codes(0, 0, n)
    compare_codes(kc, r.kc, r.kx, cal.ck, w.k_sub, "cfg1/k/all", log)
    compare_codes(vc, r.vc, r.vx, cal.cv, w.v_sub, "cfg1/v/all", log)
    write_tie_log("full_cfg1_all", log)


def test_full_size_decode_step_default_splits_llama_32k():
    """The call bench.py times, vq_decode_step with the library's split count,
    at the 32K workload's full size: every query head against the oracle.

    The cached 32768 tokens hold the oracle's own codes (written into the
    pools); the step encodes and appends token 32768 itself, so its codes are
    compared with the oracle's, and the outputs of all 32 query heads with the
    oracle's attention over all 32769 tokens."""
    w = W.WORKLOADS[1]
    cal = stored_calib(1)
    gc = GpuCache(w, cal)
    n = int(gc.lens[0])
    r = oracle_encode(w, cal, 0, 0, n + 1)
    gc.write_codes(0, 0, r.kc[:n], r.vc[:n])
    q = W.queries(w)
    got = gc.step(q)                                  # appends token n, attends over n + 1
    assert gc.device_status() == 0
    log = []
    kc, vc = gc.codes(0, n, n + 1)
    ties = compare_codes(kc, r.kc[n:], r.kx[n:], cal.ck, w.k_sub, "cfg1/step/k", log)
    ties += compare_codes(vc, r.vc[n:], r.vx[n:], cal.cv, w.v_sub, "cfg1/step/v", log)
    write_tie_log("full_cfg1_step", log)
    ref = oracle_attention(w, cal, q[0], r.kc, r.vc)
    if ties == 0:
        check_outputs(got[0], ref, "cfg1 decode step, all heads")
    else:
        skip_end_to_end("cfg1 decode step", ties)
        gc.write_codes(0, n, r.kc[n:], r.vc[n:])
        check_outputs(gc.decode(q), ref[None], "cfg1 attention on oracle codes, all heads")
