"""Reference oracle (test infrastructure only; see oracle.py)."""
from .oracle import (build, convert_f64, convert_f32, quantize, dequantize,  # noqa: F401
                     linear_mulfree, linear_dense, linear_grad_x_mulfree, linear_grad_x_dense,
                     bf16_bits_to_f64, Quantized,
                     OracleError, NonFiniteInput)
