"""GB300-native FlashAttention-2-style attention forward (placeholder; the binding follows)."""
