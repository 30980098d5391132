"""CPU f64 oracle of the blr layer: test infrastructure only (see blr_oracle)."""
from .blr_oracle import (  # noqa: F401
    adam_step,
    backward,
    backward_paths,
    backward_sampled,
    forward,
    forward_paths,
    pack_signs,
    plane_linear,
    rel_err,
    sign_grads,
    sign_grads_sampled,
    unpack_signs,
    words_per_row,
)
