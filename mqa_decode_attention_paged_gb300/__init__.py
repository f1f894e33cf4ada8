"""GB300 (sm_103a) single-query paged decode attention: MLA (primary) and GQA.

The compute path is the CUDA library ``_lib/libmqa_decode.so`` behind the C ABI
in ``include/mqa_decode.h``; this package adds a thin ctypes binding
(:mod:`._binding`), the in-tree build (:mod:`.build`) and the exchange of
decode context parallelism (:mod:`.dcp`).  Importing the binding fails
loudly when the library has not been built.  (The seeded synthetic workloads
of the tests and the benchmark live outside the package, in ``synth.py`` at
the repository root.)
"""
from .build import LIB_PATH  # noqa: F401


def _load_binding():
    import importlib
    return importlib.import_module(__name__ + "._binding")


def __getattr__(name):
    exported = {
        "mla_decode", "mla_decode_fixed_splits", "mla_decode_multi", "mla_decode_sparse", "gqa_paged_decode", "lse_merge", "num_kv_splits",
        "mla_decode_workspace_bytes", "gqa_paged_decode_workspace_bytes", "status_string", "abi_version", "device_sm_count",
        "MqaError",
    }
    if name in exported:
        return getattr(_load_binding(), name)
    raise AttributeError(name)
