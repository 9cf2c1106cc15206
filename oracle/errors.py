"""Error kinds the oracle can raise (test infrastructure, CPU oracle).

Each kind names one condition the step cannot process; tests check that the
CUDA path reports the same condition through its own status word.
"""

DEV_BAD_TOKEN = "bad_token"            # drafted token outside [0, V)
DEV_NONFINITE = "nonfinite"            # NaN or +inf logit or log-weight
DEV_EMPTY_ROW = "empty_row"            # a row whose logits are all -inf
DEV_ALL_ZERO_WEIGHT = "all_zero_weight"  # every particle of a prompt has weight 0
DEV_POOL_EXHAUSTED = "pool_exhausted"  # free block stack cannot cover the pops
DEV_TABLE_OVERFLOW = "table_overflow"  # a particle needs more than T blocks
DEV_BAD_BLOCK = "bad_block"            # block id outside the prompt's pool


class OracleError(Exception):
    """Raised by the oracle; ``kind`` is one of the DEV_* names above."""

    def __init__(self, kind, msg=""):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind
