"""Q8_0 GEMV for batch-1 / small-batch LLM decode, hand-written for GB300 (sm_103a)."""
