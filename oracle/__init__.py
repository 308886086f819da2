"""Oracle: a plain fp64 CPU restatement of the sampler and the speculative
verifier, written from the pages, used to check the CUDA path.

This package is TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and
bench.py's cpu_baseline leg (and its --impl reference arm) may import it.  It
shares no code with the CUDA library: no kernels, helpers, tables or constant
generators.  Its one shared dependency with the CUDA side is the seeded input
generator module spec_verify_gb300.workloads, which holds none of the method's
arithmetic.

Modules:
    philox   -- Philox4x64-10 and the uniform construction
    sampler  -- temperature, top-k, top-p, min-p, eq. 39.2, the id-order draw
    verify   -- accept test (eq. 39.3), residual (eq. 39.4), bonus token;
                temperature, filters and greedy verification; acceptance rates
    prepass  -- repetition penalty and constraint mask before sampling
    beam     -- one beam-search step's candidate selection (eq. 39.1)
    pool     -- runs the per-row functions above over a batch on several
                host cores (worker processes; no arithmetic of its own)
"""

from . import beam, philox, pool, prepass, sampler, verify  # noqa: F401
from .sampler import ROW_BAD_PARAMS, ROW_NONFINITE, ROW_OK  # noqa: F401
