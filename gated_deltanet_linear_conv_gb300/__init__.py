"""GB300 (sm_103a) Gated DeltaNet token mixer.

``gdn`` binds the C-ABI CUDA library libgdn.so (built by ``build()``);
``inputs`` draws the seeded synthetic workloads.  The library is loaded on
first use and its absence is an error: there is no CPU fallback.
"""

from . import gdn, inputs  # noqa: F401

__all__ = ['inputs', 'gdn', 'build']


def build(force=False):
    from . import _build
    return _build.build(force=force)
