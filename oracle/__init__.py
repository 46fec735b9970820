"""fp64 CPU oracle for soft-capped attention (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package; the CUDA library never imports, links or calls it.
"""

from .capattn_oracle import (  # noqa: F401
    OracleConfig, alsc_constants, backward, backward_kv_head, cap_derivative, cap_forward,
    config_from_workload, forward, loss, mask_matrix, mask_rows, pair_count,
    visit_matrix,
)
