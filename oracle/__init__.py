"""Plain, slow, obviously-correct CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (``paged_kv_cache_51_gb300``)
imports, links or runs this package; it shares no code, header, table or helper
with the CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may use it.

Everything is NumPy in float64 (bf16 cache values are widened exactly).  The
pages this follows are cited by title and section; the short tags are

  [Deploy]   "大模型部署.md" (AIGC-Interview-Book): §2.1 vLLM 框架技术详解
             (3. 调度策略与显存块管理; 4. PageAttention 内存管理技术详解),
             §2.5 LMDeploy (2. TurboMind), §4.1 注意力机制计算优化
             (1. FlashAttention; 4. MQA 与 GQA)
  [Infra]    "【自用】AI infra相关", 一、推理两阶段 / 二、vLLM
  [FastGen]  "DeepSpeed-FastGen 深度解析", §3 动态 SplitFuse / §6 源码
  [Ch7]      "第7章：大模型部署实战：从单机到集群的演进路径", §2.1 / §2.2
  [Ch15]     "第 15 章：推理引擎与部署", §15.1 Flash Attention 原理与实现 /
             §15.6 vLLM 高级特性与性能优化

Modules
  numerics     exact widening of cache-dtype values to float64
  attention    block-table walk + exact softmax(QK^T/sqrt(d))V (decode, varlen)
  cache        slot-mapped append and whole-block copy on a cache mirror
  block_pool   ref-counted block pool with copy-on-write and admission
  online       the tiled online-softmax recurrence and the split merge (a
               second, independent path used only to pin the first)
  sketch       the pages' per-block-normalised sketch (a negative control)
  kv_size      closed-form KV-cache size
  splitfuse    token-budget composition of one forward pass (decodes + prompt chunks)
  rope         rotate-half rotary embedding fused into the append (fp32, bf16 rounding)
  quant        8-bit KV cache: per-(token, head) symmetric int8 codes and decode over them

Parity: every function here is pinned by ``tests/test_oracle_*.py`` against
values the pages print, closed forms, brute force on unpaged data, or
invariants; none is marked "parity unpinned".
"""

from . import (attention, block_pool, cache, kv_size, numerics, online, quant, rope,  # noqa: F401
               sketch, splitfuse)
