"""Float64 CPU oracle for the fused attention backward pass.

TEST INFRASTRUCTURE ONLY. Nothing in the library imports, calls or links this
package. Only the tests, the package smoke check and the benchmark's CPU
baseline leg may use it. It shares no code with the CUDA path.

Every function is a plain NumPy restatement, in float64, of the formulas on
the source pages:
  * composable_kernel "34_bwd_gqa_fmha.py": forward with LSE, the backward
    D = rowsum(dO * O), dP = dO V^T, dS = P (dP - D), dQ = scale dS K,
    dK = scale dS^T Q, dV = P^T dO, and the GQA head-group sum of dK / dV.
  * composable_kernel "28_backward_dbias_fmha.py": elementwise bias added
    after scaling, dbias = sum over batch of P (dP - D).
  * composable_kernel "22_sink_tokens_fmha.py": causal, causal + sink and
    sliding window + sink masks.
  * Ascend "sparse_flash_mla_grad": selected-KV sparse backward with shared
    latent KV (K = V), P rebuilt from the given LSE, dKV = scale dS^T Q + P^T dO.

Pins (tests/test_oracle_*.py): central finite differences of L = sum(O * dO),
sum_j dS_ij = 0, GQA ratio 1 == MHA, GQA == expanded MHA + group sum,
closed forms (Sk = 1, constant V rows, bias constant along j), brute-force
Python loops on tiny shapes, the sparse path reducing to the dense one, and
hand-derived values in tests/golden/.
"""

from .dense import (
    causal_mask,
    causal_sink_mask,
    window_sink_mask,
    live_mask,
    forward,
    preprocess,
    dsinks,
    backward,
    varlen_forward,
    varlen_backward,
)
from .sparse import (
    selected_rows,
    sparse_forward,
    sparse_backward,
)

__all__ = [
    "causal_mask",
    "causal_sink_mask",
    "window_sink_mask",
    "live_mask",
    "forward",
    "preprocess",
    "dsinks",
    "backward",
    "varlen_forward",
    "varlen_backward",
    "selected_rows",
    "sparse_forward",
    "sparse_backward",
]
