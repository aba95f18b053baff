"""Model / step shapes of the decoder workloads this library trains.

Five shapes, each a pre-RMSNorm decoder with SwiGLU MLP, rotate-half RoPE,
grouped-query attention and untied embedding / LM head:

* ``tiny``   -- 2 layers, hidden 256, 4 heads x 64, FFN 1024, vocab 1024,
  batch 2 x seq 128 (the small case the CPU oracle finishes in seconds);
* ``1.2b``   -- 22 layers, hidden 2048, 16 x 128 heads with 4 KV heads,
  FFN 5632, vocab 32000, batch 4 x seq 2048;
* ``7.6b``   -- Qwen2.5-7B shape: 28 layers, hidden 3584, 28 x 128 heads with
  4 KV heads, FFN 18944, vocab 152064, RoPE base 1e6, 4 micro-batches of
  1 x 4096;
* ``14.7b``  -- Qwen2.5-14B shape: 48 layers, hidden 5120, 40 x 128 heads with
  8 KV heads, FFN 13824, vocab 152064, RoPE base 1e6, 4 micro-batches of
  1 x 4096;
* ``lc32k`` / ``lc128k`` / ``lc512k`` -- the 7.6B shape at batch 1 with one
  sequence of 32768 / 131072 / 524288 tokens;
* ``tiny_moe`` -- ``tiny`` with every MLP replaced by a routed mixture of 8
  SwiGLU experts (FFN 256), top-2 per token (the oracle-size MoE case);
* ``moe`` -- a GPT-OSS-style MoE decoder (the model family of the pages' MoE
  benchmark, lilting.ch MoE section): hidden 2880, 64 x 64 heads with 8 KV
  heads, 32 experts of FFN 2880 with top-4 routing, vocabulary 201088, RoPE
  base 150000, 4 micro-batches of 1 x 4096; 8 layers (7.7B parameters, so the
  host state fits the 199 GB of host RAM of one GB300 node's share).
"""
from __future__ import annotations

_COMMON = dict(rms_eps=1e-6, init_std=0.02, lr=1e-3, beta1=0.9, beta2=0.999,
               adam_eps=1e-8, weight_decay=0.0)

CONFIGS: dict[str, dict] = {
    "tiny": dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=1024,
                 vocab=1024, batch=2, seq=128, micro=1, rope_base=1e4, steps=3),
    "1.2b": dict(n_layers=22, hidden=2048, n_heads=16, n_kv_heads=4, head_dim=128, ffn=5632,
                 vocab=32000, batch=4, seq=2048, micro=1, rope_base=1e4, steps=10),
    "7.6b": dict(n_layers=28, hidden=3584, n_heads=28, n_kv_heads=4, head_dim=128, ffn=18944,
                 vocab=152064, batch=1, seq=4096, micro=4, rope_base=1e6, steps=6),
    "14.7b": dict(n_layers=48, hidden=5120, n_heads=40, n_kv_heads=8, head_dim=128, ffn=13824,
                  vocab=152064, batch=1, seq=4096, micro=4, rope_base=1e6, steps=6),
    "lc32k": dict(n_layers=28, hidden=3584, n_heads=28, n_kv_heads=4, head_dim=128, ffn=18944,
                  vocab=152064, batch=1, seq=32768, micro=1, rope_base=1e6, steps=3),
    "lc128k": dict(n_layers=28, hidden=3584, n_heads=28, n_kv_heads=4, head_dim=128, ffn=18944,
                   vocab=152064, batch=1, seq=131072, micro=1, rope_base=1e6, steps=1),
    "lc512k": dict(n_layers=28, hidden=3584, n_heads=28, n_kv_heads=4, head_dim=128, ffn=18944,
                   vocab=152064, batch=1, seq=524288, micro=1, rope_base=1e6, steps=1),
    "tiny_moe": dict(n_layers=2, hidden=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=256,
                     vocab=1024, batch=2, seq=128, micro=1, rope_base=1e4, steps=3,
                     n_experts=8, top_k=2, expert_ffn=256),
    "moe": dict(n_layers=8, hidden=2880, n_heads=64, n_kv_heads=8, head_dim=64, ffn=2880,
                vocab=201088, batch=1, seq=4096, micro=4, rope_base=1.5e5, steps=3,
                n_experts=32, top_k=4, expert_ffn=2880),
}
for _c in CONFIGS.values():
    for _k, _v in _COMMON.items():
        _c.setdefault(_k, _v)


def get(name: str, **over) -> dict:
    c = dict(CONFIGS[name])
    c.update(over)
    return c


def tokens_per_step(c: dict) -> int:
    return c["micro"] * c["batch"] * c["seq"]
