"""GB300 (sm_103a) Qwen3-style decoder forward pass behind the libqw C ABI.

``build()`` compiles the CUDA library in-tree; ``qw`` is its ctypes binding.
"""

from ._build import build as _build_lib


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile libqw.so for sm_103a (if needed) and load it."""
    path = _build_lib(verbose=verbose, force=force)
    from . import qw
    qw.load()
    return path


from . import qw  # noqa: E402,F401
