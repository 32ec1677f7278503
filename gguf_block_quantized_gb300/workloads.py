"""The benchmark and parity workloads: matrix shapes and weight formats.

Format codes are the library's own (1 = Q8_0, 2 = Q4_K, 3 = Q6_K, 4 = Q8_K, 5 = Q4_0,
6 = Q5_0, 7 = F16).
The Q4_K_M mix follows "The GGML ecosystem, and where synapse fits", section 3
(llama-quantize): most matrices Q4_K; attn_v and ffn_down Q6_K in the first and last
eighth of the layers and every third layer between them.
"""
from __future__ import annotations

from dataclasses import dataclass

Q8_0, Q4_K, Q6_K, Q8_K, Q4_0, Q5_0, F16 = 1, 2, 3, 4, 5, 6, 7
TYPE_NAMES = {Q8_0: "Q8_0", Q4_K: "Q4_K", Q6_K: "Q6_K", Q8_K: "Q8_K", Q4_0: "Q4_0", Q5_0: "Q5_0", F16: "F16"}
BLOCK_ELEMS = {Q8_0: 32, Q4_K: 256, Q6_K: 256, Q8_K: 256, Q4_0: 32, Q5_0: 32, F16: 1}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210, Q8_K: 292, Q4_0: 18, Q5_0: 22, F16: 2}


@dataclass(frozen=True)
class Matrix:
    name: str
    wtype: int
    n_out: int
    n_in: int

    @property
    def weight_bytes(self) -> int:
        return self.n_out * (self.n_in // BLOCK_ELEMS[self.wtype]) * BLOCK_BYTES[self.wtype]


def gemv_bytes(m: Matrix, n_tok: int) -> int:
    """Algorithmic bytes of one decode product: weights + fp32 activations + fp32 outputs."""
    return m.weight_bytes + 4 * m.n_in * n_tok + 4 * m.n_out * n_tok


def gemm_flops(m: Matrix, n_tok: int) -> int:
    return 2 * m.n_out * m.n_in * n_tok


# Q8_0 GEMV, 2048 x 2048, one token.
Q8_0_SQUARE = [Matrix("w", Q8_0, 2048, 2048)]

# One Llama-1B-shaped layer for decode (d = 2048, ffn = 8192, 32q/8kv heads of 64).
LLAMA1B_LAYER = [
    Matrix("attn_q", Q4_K, 2048, 2048),
    Matrix("attn_k", Q4_K, 512, 2048),
    Matrix("attn_v", Q4_K, 512, 2048),
    Matrix("attn_output", Q4_K, 2048, 2048),
    Matrix("ffn_gate", Q4_K, 8192, 2048),
    Matrix("ffn_up", Q4_K, 8192, 2048),
    Matrix("ffn_down", Q6_K, 2048, 8192),
]

# Q6_K output projection of a 128256-token vocabulary at d = 2048.
LM_HEAD_1B = [Matrix("output", Q6_K, 128256, 2048)]

# Llama-8B-shaped FFN pair for prefill.
LLAMA8B_FFN = [Matrix("ffn_up", Q4_K, 14336, 4096), Matrix("ffn_down", Q4_K, 4096, 14336)]


def use_more_bits(i_layer: int, n_layers: int) -> bool:
    """Q4_K_M rule: first and last eighth of the layers, and every third layer between."""
    lo, hi = n_layers // 8, 7 * n_layers // 8
    return i_layer < lo or i_layer >= hi or (i_layer - lo) % 3 == 2


def llama8b_q4_k_m(n_layers: int = 32, d: int = 4096, ffn: int = 14336, kv: int = 1024,
                   vocab: int = 128256, lm_head: bool = True) -> list[Matrix]:
    """Every projection of a Llama-8B-shaped model in the Q4_K_M mix (+ Q6_K lm_head)."""
    mats: list[Matrix] = []
    for i in range(n_layers):
        more = use_more_bits(i, n_layers)
        mats += [
            Matrix(f"blk.{i}.attn_q", Q4_K, d, d),
            Matrix(f"blk.{i}.attn_k", Q4_K, kv, d),
            Matrix(f"blk.{i}.attn_v", Q6_K if more else Q4_K, kv, d),
            Matrix(f"blk.{i}.attn_output", Q4_K, d, d),
            Matrix(f"blk.{i}.ffn_gate", Q4_K, ffn, d),
            Matrix(f"blk.{i}.ffn_up", Q4_K, ffn, d),
            Matrix(f"blk.{i}.ffn_down", Q6_K if more else Q4_K, d, ffn),
        ]
    if lm_head:
        mats.append(Matrix("output", Q6_K, vocab, d))
    return mats
