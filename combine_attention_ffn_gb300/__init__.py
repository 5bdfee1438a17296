"""GB300-native MoE token dispatch and combine between Attention sources and
FFN expert workers, on one GPU.

The exchange runs in hand-written sm_103a CUDA kernels behind a C ABI
(``include/afd.h``, built into ``libafd.so`` in this directory). ``afd``
is the thin Python binding over it; ``workloads`` draws seeded synthetic
inputs. Importing this package does not load the CUDA library: the first use
of :class:`Buffer` does, and fails loudly if it has not been built.
"""

__all__ = ["Buffer", "AfdError", "load_library", "route_layout_noalloc",
           "COMBINE_FUSED", "COMBINE_TWO_STAGE", "COMBINE_TWO_STAGE_FP8"]


def __getattr__(name):
    if name in __all__:
        from . import afd

        return getattr(afd, name)
    raise AttributeError(name)
