"""Stable LatentMoE feed-forward layer (forward pass) for GB300 / sm_103a.

The compute path is the C-ABI library built from csrc/ (see include/lmoe.h);
this package only loads it and marshals torch tensors into its calls."""
from .binding import (LatentMoE, LmoeError, load_library, status_string, make_config, EXPORTS,  # noqa: F401
                      LMOE_OK, LMOE_ERR_INVALID_ARG, LMOE_ERR_UNSUPPORTED, LMOE_ERR_CUDA, LMOE_ERR_OOM,
                      LMOE_ERR_TIMEOUT)
