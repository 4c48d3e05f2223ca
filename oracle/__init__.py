"""fp64 CPU oracle of the DSA hot path (test infrastructure only; see dsa_oracle)."""
from .dsa_oracle import (Problem, bf16_to_f64, e4m3_to_f64, e8m0_to_f64, indexer_row,
                         mx_dequant, problem_from_case, query_rows, sfa_row, to_f64, topk_row,
                         torch_case_arrays)
