"""GB300-native FlashAttention-2 forward (placeholder; binding added with the C-ABI)."""
