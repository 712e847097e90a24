"""Pure-Python scalar-loop evaluation of the same definitions, for tiny inputs.

TEST INFRASTRUCTURE ONLY.  A second, independent transcription used to
cross-check :mod:`oracle.lssar_oracle` on L <= 32: plain ``math`` and
loops, no NumPy, no rescaling tricks (``ReLU(i*a - O)**p`` is raised
directly, which is safe for the small i and p used here), and softplus as
the literal ``log(1 + exp(x))``.  Same readings as the NumPy oracle:
natural log, 1-based i, L2 norm clamped at 1e-12, O = 0 on rows 1-3, and an
all-zero re-weighted row read as the uniform prefix mean.
"""

import math

MODE_SOFTMAX = 0
MODE_LSSA = 1
MODE_LSSAR = 2
MODE_SOFTMAX_RW = 3
MODE_SIGMOID_RW = 4


def _dot(a, b):
    return sum(x * y for x, y in zip(a, b))


def attention_bruteforce(q, k, v, mode, p=3, o_override=None):
    """q, k, v: L x d nested lists (one head).  Returns the L x d output."""
    L = len(q)
    d = len(q[0])
    out = []
    for i in range(1, L + 1):
        qi = q[i - 1]
        if mode in (MODE_SOFTMAX, MODE_SOFTMAX_RW):
            sc = [_dot(qi, k[j]) / math.sqrt(d) for j in range(i)]
            top = max(sc)
            e = [math.exp(s - top) for s in sc]
            z = sum(e)
            a = [x / z for x in e]
        else:
            nq = max(math.sqrt(_dot(qi, qi)), 1e-12)
            c = math.log(d) * math.log(i)
            a = []
            for j in range(i):
                nk = max(math.sqrt(_dot(k[j], k[j])), 1e-12)
                cos = _dot(qi, k[j]) / (nq * nk)
                if mode == MODE_SIGMOID_RW:
                    a.append(1.0 / (1.0 + math.exp(-c * cos)))
                else:
                    a.append(math.log(1.0 + math.exp(c * cos)))
            z = sum(a)
            a = [x / z for x in a]
        if mode in (MODE_LSSAR, MODE_SOFTMAX_RW, MODE_SIGMOID_RW):
            o = (0.0 if i <= 3 else 1.0) if o_override is None else float(o_override)
            # ReLU; residues of 0 left by rounding (at most 1e-10) are 0
            r = [(i * x - o) ** p if i * x - o > 1e-10 else 0.0 for x in a]
            t = sum(r)
            w = [x / t for x in r] if t > 0.0 else [1.0 / i] * i
        else:
            w = a
        out.append([sum(w[j] * v[j][t] for j in range(i)) for t in range(d)])
    return out
