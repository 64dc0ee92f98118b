"""GB300-native M²RNN forward recurrence: a C-ABI CUDA library (libm2rnn.so) and its
thin Python binding.  Importing the package does not load the library; the first
call does, and raises if it has not been built."""
from .m2rnn import (M2RNNError, load_library, m2rnn_forward, m2rnn_forward_bf16,  # noqa: F401
                    m2rnn_forward_bf16_variant, m2rnn_forward_f32, pick_variant,
                    status_string, stream_status, variant_name, variant_supports,
                    version)
