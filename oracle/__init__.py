"""FP64 CPU oracle for normalised causal linear attention (forward and its
gradients) and the delta-rule memory (test infrastructure).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The product library never links, loads or calls it, and this package
imports nothing from the product.
"""
from .oracle import (  # noqa: F401
    PHI_ELU1,
    PHI_IDENTITY,
    PHI_RELU1,
    backward,
    build,
    chunkwise,
    delta,
    dense,
    num_cpus,
    scan,
    variant,
)
