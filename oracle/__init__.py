"""Reference oracle for the attention library's parity tests.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, the smoke check and the
benchmark's CPU-baseline leg, never by the library itself.
"""

from .mqa import (  # noqa: F401
    attention, block_status, pad_rows, pair_visibility, raw_visible, comp_visible,
    padded_lengths, ceil_to, H, D, BLOCK,
)
from . import indexer  # noqa: F401,E402
from . import fp8  # noqa: F401,E402
from . import compressor  # noqa: F401,E402
