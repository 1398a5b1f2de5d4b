"""GB300-native fused attention forward (sm_103a).

``O = softmax(scale * Q K^T + mask) V`` with online softmax, fp32 LSE, split-KV
partials merged by LSE, MHA/MQA/GQA, head dims 64/128/256/512, decode and short
prefill, sliding-window and bottom-right causal masks.

Every step runs in the CUDA kernels of ``libfmha_gb300.so`` behind a C ABI
(``include/fmha.h``).  ``binding`` marshals torch tensors into that ABI; there
is no CPU fallback: if the library is missing the calls raise.
"""
from . import inputs  # noqa: F401  (shapes and seeded random inputs only)


def __getattr__(name):
    # The binding loads the shared library on first use, so that importing the
    # package for its input generators needs neither a GPU nor a built library.
    if name in ("binding",):
        import importlib
        return importlib.import_module("." + name, __name__)
    from . import binding
    try:
        return getattr(binding, name)
    except AttributeError:
        raise AttributeError(name) from None
