"""Seeded synthetic inputs for the NAtS-L hybrid attention layer forward.

This package is shared by the CUDA path's tests and benchmark and by the
oracle's tests.  It holds random draws and input construction only (rounding
to the storage dtype, unit-norm keys, the planted chunk structure that the
score layer later recovers); none of the layer's own arithmetic lives here.
"""

from .synth import (  # noqa: F401
    NatsInputs,
    CONFIGS,
    config_inputs,
    make_inputs,
    round_to_bf16,
    bf16_bits,
    NatsXInputs,
    X_CONFIGS,
    make_x_inputs,
    x_config_inputs,
    NhaInputs,
    NHA_CONFIGS,
    make_nha_inputs,
    nha_config_inputs,
)
