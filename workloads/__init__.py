"""Seeded synthetic inputs for paged-attention forward.

This package draws inputs and builds block tables / cumulative lengths; it
holds none of the attention arithmetic.  Both the CUDA path (through the
binding) and the oracle consume what it produces, so the two see identical
bits.
"""
from .synth import (  # noqa: F401
    DecodeCase,
    VarlenCase,
    decode_config,
    make_decode,
    make_varlen,
    to_numpy,
    varlen_config,
    CONFIG_NAMES,
)
