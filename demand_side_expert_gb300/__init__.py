"""GB300-native recalibrated MoE expert backward (LRMoE hot path, one GPU).

The compute path is liblrm.so (hand-written CUDA for sm_103a, C ABI in
include/lrm.h); ``lrm`` is its ctypes binding and ``pipeline`` the host-side
buffer owner that issues the calls in order. Touching either requires the
built library (``python -m demand_side_expert_gb300.build``); there is no
fallback implementation. The submodules load lazily so that the build step
itself can be imported before the library exists.
"""

_LAZY = {
    "lrm": ("lrm", None),
    "pipeline": ("pipeline", None),
    "RecalibratedExpertBackward": ("pipeline", "RecalibratedExpertBackward"),
    "dtype_code": ("pipeline", "dtype_code"),
}


def __getattr__(name):
    if name not in _LAZY:
        raise AttributeError(name)
    import importlib

    mod_name, attr = _LAZY[name]
    mod = importlib.import_module(f"{__name__}.{mod_name}")
    return mod if attr is None else getattr(mod, attr)
