"""The partition's length-penalty weight lambda = mean curvature, summed in
the order kvc_partition uses, so that the GPU tests can hand the oracle's
dynamic program the same lambda bit for bit.

kvc_partition's CTA of 512 threads sums kappa[0:end) in float64: thread i
adds kappa[i], kappa[i + 512], ... in increasing order starting from 0.0,
then the 512 partial sums are combined pairwise with a halving stride
(part[i] = part[i] + part[i + h] for h = 256, 128, ..., 1), and the total is
divided by end.  The lambda of the GraceKV "01 Curvature-guided partition"
reading is the plain mean; only the rounding order is fixed here.
"""
import numpy as np

THREADS = 512


def partition_lambda(kappa_row, end):
    k = np.asarray(kappa_row[:end], np.float64)
    part = [0.0] * THREADS
    for t in range(end):
        part[t % THREADS] += float(k[t])
    h = THREADS // 2
    while h:
        for i in range(h):
            part[i] = part[i] + part[i + h]
        h //= 2
    return part[0] / end
