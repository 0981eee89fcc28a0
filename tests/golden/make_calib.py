"""Write the offline calibration of every workload: smoothing factors and codebooks.

Calls only the oracle (and the seeded workload generators).  For each workload
it draws the 16384-token calibration set, computes lambda per KV head
(VecInfer, 方法细节 "异常值抑制的向量量化": lambda_i = sqrt(max |K_i|)), transforms
the calibration keys (K diag(lambda)^-1 H_D), and runs 10 Lloyd iterations from a
seeded choice of distinct training rows on the pooled sub-vectors of all heads:
transformed keys for C_k, raw values for C_v (VecInfer, "注意力机制中的向量量化
KV缓存": codebooks pre-trained offline with K-Means).  lambda is stored as fp32,
the codebooks as fp16 (2 bytes per centroid element, as the page counts them).

    python tests/golden/make_calib.py [workload index ...]
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "calib")


def calibrate(w):
    k_cal, v_cal = workloads.calibration(w)
    lam = oracle.smoothing_lambda(k_cal).astype(np.float32)
    kt = oracle.transform_keys(k_cal, lam.astype(np.float64))
    xk = kt.reshape(-1, w.k_sub)
    xv = v_cal.astype(np.float64).reshape(-1, w.v_sub)
    ck, obj_k = oracle.kmeans(xk, workloads.kmeans_init(len(xk), 2 ** w.k_bits, "k"),
                              workloads.KMEANS_ITERS)
    cv, obj_v = oracle.kmeans(xv, workloads.kmeans_init(len(xv), 2 ** w.v_bits, "v"),
                              workloads.KMEANS_ITERS)
    return dict(lam=lam, ck=ck.astype(np.float16), cv=cv.astype(np.float16),
                obj_k=obj_k, obj_v=obj_v)


def path(i):
    return os.path.join(OUT, f"cfg{i}.npz")


def main(argv):
    os.makedirs(OUT, exist_ok=True)
    idx = [int(a) for a in argv] or sorted(workloads.WORKLOADS)
    for i in idx:
        w = workloads.WORKLOADS[i]
        c = calibrate(w)
        np.savez(path(i), **c)
        print(f"cfg{i} {w.name}: lambda {c['lam'].shape}, C_k {c['ck'].shape}, "
              f"C_v {c['cv'].shape}, objective K {c['obj_k'][0]:.4g}->{c['obj_k'][-1]:.4g}, "
              f"V {c['obj_v'][0]:.4g}->{c['obj_v'][-1]:.4g}", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
