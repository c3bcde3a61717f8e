"""CPU oracle of the GDN speculative-decoding hot path -- test infrastructure only.

Importable by the tests, the smoke check and the bench's CPU-baseline leg; never by the
library.  See ``gdn_ref.c`` for what it computes and the passages it follows.
"""
from .gdn_ref import Layer, Rows, build, build_all, conv_update, mixed_batch, recurrent  # noqa: F401
