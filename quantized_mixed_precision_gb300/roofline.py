"""Work and traffic accounting for the roofline figures.

The model is the one the JAX Pallas TPU matmul tutorial uses in its section
矩阵乘法性能分析: a matmul of (m, k) by (k, n) does 2*m*k*n operations and
must move at least (m*k + k*n + m*n) * itemsize bytes.  Here every operand
carries its own width in bits, so packed 4-bit and 2-bit weights count 0.5
and 0.25 bytes per element, and per-row / per-column scale vectors are added.
"""


def matmul_ops(m, k, n):
    return 2 * m * k * n


def matmul_min_bytes(m, k, n, a_bits, b_bits, c_bits, extra_bytes=0):
    bits = m * k * a_bits + k * n * b_bits + m * n * c_bits
    return bits // 8 + extra_bytes


def quantize_bytes(rows, cols, x_bits=16, q_bits=8):
    """Read x once, write the codes and one fp16 scale per row."""
    return (rows * cols * (x_bits + q_bits)) // 8 + 2 * rows
