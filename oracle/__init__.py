"""Float64 CPU oracle for causal LSSAR / LSSA / softmax attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
legs of ``bench.py`` use it.  It shares no code with the CUDA path.

Source of truth: the papernotes.org notes on "Softplus Attention with
Re-weighting Boosts Length Extrapolation in Large Language Models"
(arXiv 2501.13428), sections "Method details / overall framework" and
"Key design 1-3", plus the scaled dot-product formula in "Background".
"""

from .lssar_oracle import (  # noqa: F401
    MODE_SOFTMAX,
    MODE_LSSA,
    MODE_LSSAR,
    MODE_SOFTMAX_RW,
    MODE_SIGMOID_RW,
    softplus,
    sigmoid,
    l2_normalize_rows,
    length_scale,
    bias_o,
    lssa_rows,
    reweight_rows,
    attention_rows,
    attention_forward,
)
from .bruteforce import attention_bruteforce  # noqa: F401
from .lssar_backward import attention_backward, head_backward  # noqa: F401
