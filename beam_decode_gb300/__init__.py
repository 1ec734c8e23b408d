"""GB300-native wide-beam semantic-ID decode step.

The compute path is libgrbeam (CUDA, sm_103a) behind the C ABI in
include/grbeam.h; ``binding`` is its thin ctypes layer and ``workload`` the
seeded synthetic inputs.
"""
from . import binding, workload  # noqa: F401
from .binding import Beam, GrError, Trie  # noqa: F401
