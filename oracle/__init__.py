"""Oracle (test infrastructure only): plain CPU restatement of the MoE layer forward.

Only the tests, the smoke check and the bench's CPU-baseline leg import this package.
"""
from . import attention_oracle, moe_oracle  # noqa: F401
