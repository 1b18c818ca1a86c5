"""Block-scaled FP4 (E2M1) codec for GB300 (sm_103a)."""
