"""Small-M FP8 block-scaled linear layer for GB300 (sm_103a)."""
