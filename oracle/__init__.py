"""fp64 CPU oracle (test infrastructure only; see ``kd_oracle`` and ``kd_cache_oracle``)."""
from .kd_cache_oracle import topk_cache_naive, topk_cache_oracle
from .kd_oracle import kd_oracle, kd_oracle_dW_rows, kd_oracle_naive, kd_oracle_rows, valid_rows

__all__ = ["kd_oracle", "kd_oracle_naive", "kd_oracle_rows", "kd_oracle_dW_rows", "valid_rows",
           "topk_cache_oracle", "topk_cache_naive"]
