"""fp64 CPU oracle for exact scaled-dot-product attention. TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU
baseline and its ``--impl reference`` arm) may import anything from here. The
CUDA library never calls it, and it shares no code with the CUDA library: it
reads raw bf16 bit patterns and plain numpy arrays only.

What it computes is the plain definition that the tiled GPU method reaches
exactly (up to rounding order), written out with no blocking, fusion or
reordering beyond what that definition states. Sources, cited by page title
and section:

  [MG-A] menggq.pages.dev, "Transformer 架构的数学与计算深度解析：注意力机制的
         详尽研究报告" -- §2.2 scores, §2.3 scaling, §2.4 softmax and weighted
         sum, §4.1 causal mask, §4.2 cross-attention, §6.3 online softmax.
  [MG-B] menggq.pages.dev, "Transformer 深度进阶：从矩阵视角到 FlashAttention
         工程优化" -- §2.1 heads, §3.2 online-softmax update formulas, §4 shapes.
  [AUT]  auturnal.com, "从注意力到 IO 感知执行：Transformer 的计算结构、复杂度与
         可复核分析" (v10) -- §4/§6 score-matrix bytes, §8 with its first two
         equations (m, l, u recurrence), §9 with its third equation (KV cache).
  [IMR]  imreese.github.io, "Transformer 笔记：注意力机制为什么会变成系统问题" --
         the masking section (token t sees positions not later than t) and the
         prefill/decode section (decode reads cached K/V).
  [PW]   pwwt.cn news 6124947 (Transformer algorithm-evolution article) --
         §2.1 S = QK^T/sqrt(d_k), §2.3 MQA/GQA, §3.1-3.2 KV cache and its
         size, §4.2 online softmax is exact, §5.3 RoPE, §6.1 sliding window.

Parity status: every public function here is pinned by ``tests/test_oracle_pins.py``
against facts other than itself (closed forms, invariants, the pages' worked
numbers, brute force on tiny inputs, and an independent library routine).
"""
from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    attention_forward,
    attention_decode,
    attention_backward,
    attention_decode_paged,
    attention_forward_rope,
    rope_rotate,
    round_to_bf16,
    online_attention_rows,
    merge_two_blocks,
    score_bytes,
    kv_cache_bytes,
)
