"""CPU oracle for the DSA decode step -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it: the oracle has its own E4M3 / E2M1 / E8M0 / bf16
decoders, its own page translation and its own arithmetic, all in float64
(numpy) unless the method itself fixes a precision.

What it computes, and where the method is stated (page title, then section):

* "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持" (vLLM's Kimi K3.1 Pro article),
  section "K3.1 Pro 中的稀疏注意力" (sparse attention in K3.1 Pro): a small
  indexer keeps one FP8 key per token (132 B with its scale) and scores every
  earlier token with 32 light heads; the top 2,048 tokens are kept; MLA
  attention then runs exactly over those tokens only. Dense MLA reads the
  576-B FP8 latent of every context token.
* same article, section "面向三种状态的 KV 缓存" (a KV cache for three kinds
  of state): latent 576 B (FP8) or 352 B (NVFP4); index key 132 B (FP8) or
  68 B (MXFP4); kernels read the cache through per-step page addresses
  derived from the block table.
* same article, section "低延迟解码：融合的 DSA 解码路径" (fused DSA decode
  path): the indexer query is quantised to FP8 (or MXFP4) with the scale
  folded into the head weights; the scorer and an exact top-k selection are
  separate steps.
* same article, section "长上下文：带稀疏 indexer 的 decode 上下文并行"
  (decode context parallelism): partial attention outputs are merged by
  log-sum-exp.

Readings of points the pages leave open are listed in the docstrings of the
functions that take them.

Parity status per function: every public function of ``oracle.dsa`` is
pinned by a ``-m "not gpu"`` test against something other than itself (spec
values, closed forms, brute force, a library routine), except the end-to-end
composition on full-size inputs, whose only pins are those of its parts.
"""
