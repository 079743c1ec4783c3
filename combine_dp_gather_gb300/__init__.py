"""GB300-native MoE layer between DP attention and expert parallelism."""
