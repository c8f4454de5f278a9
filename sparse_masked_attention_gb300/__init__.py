"""FlashMask-style column-wise sparse masked attention for GB300 (sm_103a)."""
