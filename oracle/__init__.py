"""fp64 CPU oracle of the M²RNN forward recurrence, its backward pass, and the block's
conv/SiLU prologue and gate/RMSNorm epilogue (test infrastructure only).

Imported by the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; never by the CUDA library or its Python binding.
"""
from .m2rnn_backward import m2rnn_backward, m2rnn_backward_inputs  # noqa: F401
from .m2rnn_block import causal_conv1d, conv_silu, gate_rmsnorm, silu  # noqa: F401
from .m2rnn_oracle import (forget_gate, m2rnn_forward, m2rnn_forward_inputs,  # noqa: F401
                           m2rnn_forward_scalar, softplus)
