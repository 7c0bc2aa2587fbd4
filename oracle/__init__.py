"""fp64 CPU oracle (test infrastructure only; see ``kd_oracle``)."""
from .kd_oracle import kd_oracle, kd_oracle_naive, kd_oracle_rows, valid_rows

__all__ = ["kd_oracle", "kd_oracle_naive", "kd_oracle_rows", "valid_rows"]
