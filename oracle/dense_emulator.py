"""Dense emulator of lazy Adam -- TEST INFRASTRUCTURE, tiny tables only.

A pure-Python loop over *every* coordinate at *every* step, with no last_step
bookkeeping at all, written from "Module sparse_optimizer" (optirs-gpu 0.3.2
docs), section "Lazy Adam":

* a coordinate touched at step t gets the Adam recursion with its gradient and
  bias correction by the global step t;
* DormancyDecay: a coordinate NOT touched at step t gets what dense Adam would
  do with an explicit zero gradient to its moments -- m *= beta1, v *= beta2,
  one factor per elapsed step -- and no parameter update (lazy Adam performs no
  update on dormant steps);
* Lazy: a coordinate not touched gets nothing.

The oracle instead jumps over dormant steps with beta**gap; the two must agree.
``dense_adam`` is textbook dense Adam (every coordinate updated every step,
zero gradient where untouched) for the "parameter trajectory differs" pin.
"""
from __future__ import annotations

import math


def lazy_adam_dense(p, touches, *, lr, beta1, beta2, eps, mode):
    """p: list of floats (initial parameters).  touches: list over steps t = 1..T of
    dicts {coordinate: gradient}.  Returns (p, m, v) after T steps, all fp64 lists."""
    n = len(p)
    p = [float(x) for x in p]
    m = [0.0] * n
    v = [0.0] * n
    for t, touched in enumerate(touches, start=1):
        bc1 = 1.0 - beta1 ** t
        bc2 = 1.0 - beta2 ** t
        for i in range(n):
            if i in touched:
                g = float(touched[i])
                m[i] = beta1 * m[i] + (1.0 - beta1) * g
                v[i] = beta2 * v[i] + (1.0 - beta2) * g * g
                p[i] = p[i] - lr * (m[i] / bc1) / (math.sqrt(v[i] / bc2) + eps)
            elif mode == "dormancy_decay":
                m[i] = beta1 * m[i]
                v[i] = beta2 * v[i]
    return p, m, v


def dense_adam(p, touches, *, lr, beta1, beta2, eps):
    """Dense Adam: every coordinate updated at every step, gradient 0 where untouched."""
    n = len(p)
    p = [float(x) for x in p]
    m = [0.0] * n
    v = [0.0] * n
    for t, touched in enumerate(touches, start=1):
        bc1 = 1.0 - beta1 ** t
        bc2 = 1.0 - beta2 ** t
        for i in range(n):
            g = float(touched.get(i, 0.0))
            m[i] = beta1 * m[i] + (1.0 - beta1) * g
            v[i] = beta2 * v[i] + (1.0 - beta2) * g * g
            p[i] = p[i] - lr * (m[i] / bc1) / (math.sqrt(v[i] / bc2) + eps)
    return p, m, v


def sparse_sgd_dense(p, touches, *, lr, momentum, weight_decay):
    """Sparse SGD on a dense loop: only touched coordinates move; buffers of dormant ones stay."""
    n = len(p)
    p = [float(x) for x in p]
    buf = [0.0] * n
    for touched in touches:
        for i in range(n):
            if i in touched:
                gd = float(touched[i]) + weight_decay * p[i]
                if momentum != 0.0:
                    buf[i] = momentum * buf[i] + gd
                    p[i] = p[i] - lr * buf[i]
                else:
                    p[i] = p[i] - lr * gd
    return p, buf
