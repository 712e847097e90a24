"""GB300-native causal LSSAR attention forward (sm_103a, tcgen05/TMEM/TMA).

The CUDA library is loaded lazily on the first call, so the input generator
(`lssar_attn_fwd_gb300.inputs`) can be imported without a GPU or a build.
"""

from .inputs import MODE_LSSA, MODE_LSSAR, MODE_SIGMOID_RW, MODE_SOFTMAX, MODE_SOFTMAX_RW  # noqa: F401


def __getattr__(name):
    if name in ("lssar_attn_fwd", "lssar_attn_fwd_simt", "load_library", "device_error_word",
                "LssarError"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
