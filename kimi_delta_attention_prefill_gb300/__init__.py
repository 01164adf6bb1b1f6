"""GB300-native Kimi Delta Attention (KDA) prefill / decode."""
