"""ReplaySSM decode for GB300: a C-ABI CUDA library (librssm) plus this thin
Python binding. The kernels live in ``csrc/``; ``binding`` exposes the C calls
under their own names; ``inputs`` draws seeded synthetic workloads;
``state`` allocates the device buffers a decode session needs.
"""
from . import binding  # noqa: F401
from .binding import check, load  # noqa: F401
