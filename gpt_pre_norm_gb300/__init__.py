"""GB300-native GPT-2 pre-norm forward: C-ABI CUDA library plus a thin binding."""
