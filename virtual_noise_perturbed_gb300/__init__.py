"""Virtual-noise evolution strategies on one GB300 (sm_103a).

The population ES step of the EvoX API page
"evox.triton_kernels.kernels.virtual_noise" -- the perturbed linear forward,
the weight / bias gradient estimates, the noise dump and the mean-abs metric --
as a C-ABI CUDA library (``libvn.so``, declared in ``include/vn.h``) with a thin
Python binding. The noise is regenerated on the fly from (seed, element index)
and never materialised.
"""

from .api import (  # noqa: F401
    VNError,
    centered_ranks,
    compute_offsets,
    device_status,
    es_update,
    gradient_update,
    hash_probe,
    noise_dump,
    perturbed_linear_path,
    virtual_bias_gradient,
    virtual_flat_gradient,
    virtual_perturbed_linear,
    virtual_perturbed_mlp,
    virtual_reduce_metric,
    virtual_weight_gradient,
)

__all__ = [
    "VNError", "centered_ranks", "compute_offsets", "device_status", "es_update", "gradient_update", "hash_probe", "noise_dump", "perturbed_linear_path",
    "virtual_bias_gradient", "virtual_flat_gradient", "virtual_perturbed_linear", "virtual_perturbed_mlp",
    "virtual_reduce_metric",
    "virtual_weight_gradient",
]
