"""CPU oracle of the draft-head propose forward: test infrastructure only.

Only the tests, the package smoke check and the bench's CPU-baseline leg may
import this package; the product path never does.
"""
from .draft_head import (DraftHeadOracle, OracleError, PagePool, attention, bitmask_allowed,
                         e2m1_value, e4m3_codes, e4m3_value, nvfp4_dequant, rms_norm, rope,
                         round_bf16, select_drafts, silu, yarn_attention_factor, yarn_inv_freq)

__all__ = ["DraftHeadOracle", "OracleError", "PagePool", "attention", "bitmask_allowed",
           "e2m1_value", "e4m3_codes", "e4m3_value", "nvfp4_dequant", "rms_norm", "rope",
           "round_bf16", "select_drafts", "silu", "yarn_attention_factor", "yarn_inv_freq"]
