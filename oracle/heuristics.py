"""Minibatch (overlap-granularity) floor, reference (test infrastructure only).

The pages give the heuristic in words -- at least two full SM waves per
expert-grouped GEMM, which for the Kimi-2.5 shape is 2,368 tokens (*Cursor
Open-Sources Mixture-of-Kittens (MoK)*, "Three design decisions that
matter", overlap-granularity paragraph) -- and as a formula in the wiki note
(*Mixture-of-Kittens: our open-source MoE megakernel for NVL72s*, section
"2. 計算と通信のオーバーラップ(ミニバッチ)").  The printed formula has its
fraction upside down (it would give far less than one token).  Read as two
waves of 128 x 256 output tiles over the narrower of the two grouped GEMMs
(N = 2I for W1|W3, N = H for W2):

    M >= 2 * C * 128 * 256 / min(2I, H)

With H = 7168, I = 2048 and C = 148 SMs this is exactly 2,368.
"""

from __future__ import annotations


def minibatch_floor(H, I, num_sms, tile_m=128, tile_n=256, waves=2):
    """Smallest routed-row count that fills ``waves`` waves of output tiles."""
    return waves * num_sms * tile_m * tile_n / min(2 * I, H)
