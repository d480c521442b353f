"""GB300-native generation-pass hot path of NEO-unify: a C-ABI CUDA library and its binding."""
