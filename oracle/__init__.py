"""CPU oracle for the virtual-noise evolution-strategies step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call, link or
execute this package: only the test suite, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it. It shares no code, table, constant generator or helper
with the CUDA library; it is written from the EvoX API page
"evox.triton_kernels.kernels.virtual_noise" alone.

Modules
-------
``splitmix``  the splitmix64 finalizer, the per-(seed, index) state and the
              centered-uniform noise value, twice: once with Python integers
              (the reference definition, one element at a time) and once with
              numpy ``uint64`` arrays (bulk work; wraps mod 2**64 and shifts
              logically, as the page requires).
``es``        the method itself: the noise dump, ``compute_offsets``, the
              perturbed linear forward, the weight / bias gradient estimates,
              the mean-abs reduction metric, the centered ranks and the
              parameter update, all in float64 with the noise materialised
              explicitly; the bf16 model of the tensor-core forward (the perturbed
              weight, and optionally the output, rounded to bfloat16) and the
              floor that rounding sets on any bf16 implementation's deviation; the dump, the gradient and the forward also with the
              Gaussian variant of the noise (Box-Muller on the finalizer's
              two halves, ``splitmix.gaussian_*``).

Readings of the page (where it is silent or ambiguous) are stated in the
docstring of the function that takes them. Parity status: every function here
is pinned by a ``-m "not gpu"`` test against something other than itself
(closed forms, an independently derived inverse of the hash, the page's worked
example for ``compute_offsets``, brute force on tiny shapes, statistical
properties the page states). The seed/index mixing is a reading of the page
(it prints no noise values), so agreement with EvoX's own numbers is not
claimed anywhere.
"""

from . import splitmix, es  # noqa: F401
