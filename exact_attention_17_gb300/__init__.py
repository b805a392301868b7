"""GB300-native FlashAttention-2 forward (sm_103a)."""
