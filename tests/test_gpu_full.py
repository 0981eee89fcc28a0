"""Parity at the workloads' full sizes, in the launch configuration bench.py times.

For each workload (32K, ragged paged batch, 196K with drift, batch-64 GQA-5 with
9-bit values): the whole cache is encoded on the GPU (prefill plus the appended
token) and decoded with the library's default split count and launch shape.
The oracle then checks sampled outputs one by one:
  - codes of a window of tokens and of the appended token, for sampled
    (sequence, KV head) pairs: bit-exact except in-band ties (logged);
  - the G attention output rows of those pairs, against the fp64 oracle over
    all N + 1 tokens of the GPU's codes (which isolates the attention kernel
    from encode ties), within max-abs 2e-3 / mean-abs 2e-4.
"""
import numpy as np
import pytest

import workloads as W
from vqcase import (GpuCache, check_outputs, compare_codes, oracle_attention, oracle_encode,
                    stored_calib, write_tie_log)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

WINDOW = 256


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
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
    pairs = {(int(rng.integers(w.batch)), int(rng.integers(w.num_kv_heads))) for _ in range(2)}
    pairs.add((w.batch - 1, w.num_kv_heads - 1))
    log, ties = [], 0
    for b, h in sorted(pairs):
        n = int(gc.lens[b]) + 1                      # cached tokens + the appended one
        s0 = int(rng.integers(0, max(n - 1 - WINDOW, 1)))
        for lo, hi in ((s0, min(s0 + WINDOW, n - 1)), (n - 1, n)):
            r = oracle_encode(w, cal, b, lo, hi, heads=[h])
            kc, vc = gc.codes(b, lo, hi, heads=[h])
            ties += compare_codes(kc, r.kc, r.kx, cal.ck, w.k_sub, f"cfg{cfg}/k/b{b}h{h}/{lo}", log)
            ties += compare_codes(vc, r.vc, r.vx, cal.cv, w.v_sub, f"cfg{cfg}/v/b{b}h{h}/{lo}", log)
        kc, vc = gc.codes(b, 0, n, heads=[h])
        ref = oracle_attention(w, cal, q[b, h * G:(h + 1) * G], kc, vc, heads=[h])
        check_outputs(got[b, h * G:(h + 1) * G], ref, f"cfg{cfg} b{b} kv-head {h} ({n} tokens)")
    write_tie_log(f"full_cfg{cfg}", log)
