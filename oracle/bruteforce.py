"""Pure-Python brute force for tiny AttnRes cases (a pin for the C oracle).

TEST INFRASTRUCTURE ONLY. It is written independently of ``attnres_oracle.c``
so that the two can check each other on tiny shapes:

* sums use ``math.fsum`` (correctly rounded), not running fp64 sums;
* the depth softmax is evaluated as alpha_i = 1 / sum_j exp(e_j - e_i),
  which needs no max subtraction and shares no intermediate with the oracle;
* Block AttnRes is simulated as the stateful sublayer-by-sublayer process the
  pages describe (a list of frozen block summaries plus one running sum that
  is frozen at each block boundary), not through closed-form sums.

Definitions followed: DepthBench reading notes section 2.3 (Appendix A) for a
read; LLMRes blog "Kimi AttnRes" for the key-only RMSNorm; DepthBench reading
notes section 2.5 and the datacamp explainer ("block attention residuals") for
the block source set (embedding, frozen block sums, current running sum).
"""
from __future__ import annotations

import math


def rmsnorm_key(v, gamma, eps):
    d = len(v)
    ms = math.fsum(x * x for x in v) / d
    r = math.sqrt(ms + eps)
    return [g * x / r for g, x in zip(gamma, v)]


def read(sources, w, gamma, eps):
    """One read: (z, log-sum-exp of the scores). sources: list of lists."""
    e = [math.fsum(wk * kk for wk, kk in zip(w, rmsnorm_key(v, gamma, eps))) for v in sources]
    alpha = [1.0 / math.fsum(math.exp(ej - ei) for ej in e) for ei in e]
    d = len(sources[0])
    z = [math.fsum(a * v[k] for a, v in zip(alpha, sources)) for k in range(d)]
    lse = e[0] + math.log(math.fsum(math.exp(ej - e[0]) for ej in e))
    return z, lse


def full_pass(history, W, Gamma, eps):
    """history: list of R source vectors (one token); read r sees history[:r+1]."""
    return [read(history[: r + 1], W[r], Gamma[r], eps)[0] for r in range(len(W))]


def block_pass(embedding, outputs, S, W, Gamma, eps):
    """Sublayer-by-sublayer Block AttnRes for one token.

    outputs[k] is the output f_k of sublayer k; S sublayers form a block.
    """
    frozen = []          # completed block summaries b_1, b_2, ...
    running = None       # running sum of the current block, None while empty
    result = []
    for k, f in enumerate(outputs):
        srcs = [embedding] + frozen + ([running] if running is not None else [])
        result.append(read(srcs, W[k], Gamma[k], eps)[0])
        running = list(f) if running is None else [math.fsum((a, b)) for a, b in zip(running, f)]
        if (k + 1) % S == 0:
            frozen.append(running)
            running = None
    return result
