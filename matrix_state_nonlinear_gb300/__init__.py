"""GB300-native M²RNN forward recurrence: a C-ABI CUDA library and its Python binding."""
