"""GB300-native M²RNN recurrence (forward, and the backward for training): a C-ABI
CUDA library (libm2rnn.so) and its thin Python binding.  Importing the package does
not load the library; the first call does, and raises if it has not been built."""
from .m2rnn import (M2RNNError, backward_workspace_bytes, conv_silu, gate_rmsnorm,  # noqa: F401
                    load_library,
                    m2rnn_backward, m2rnn_decode_step, m2rnn_forward, m2rnn_forward_bf16,
                    m2rnn_forward_bf16_variant, m2rnn_forward_conv, m2rnn_forward_f32,
                    m2rnn_forward_train,
                    pick_variant,
                    status_string, stream_status, variant_name, variant_supports,
                    version)
