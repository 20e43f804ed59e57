"""fp64 CPU oracle for CSA / HCA hybrid compressed attention.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import it. It shares no code with the CUDA library.

Parity status of each function (what pins it, see tests/test_oracle_pins.py):
  bf16_to_f64, f64_to_bf16_rne   pinned: hand-worked values + exact rational rounding
  e2m1_unpack, ue8m0_to_f64      pinned: OCP MX code table fixture + bit-field decode
  compress / pooling_weights     pinned: closed forms (m=1 identity, equal logits = mean,
                                 m=2 logistic weights, weights sum to 1)
  index_scores                   pinned: brute-force integer arithmetic on nibbles + worked example
  topk_select                    pinned: brute force on tiny rows with forced ties
  attend / csa / hca layers      pinned: reduction to causal attention (m=1, k>=N, W=0),
                                 k>=E equals dense, window-only equals sliding-window attention,
                                 softmax rows sum to 1
  The index-score formula itself (ReLU per head, unit head weights) is a reading the pages do
  not print: parity unpinned for that reading.
"""
from .csa_oracle import *  # noqa: F401,F403
