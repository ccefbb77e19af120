"""GB300 FlashAttention: exact tiled attention forward and backward for sm_103a."""
