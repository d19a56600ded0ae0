"""CPU oracle for the batch-invariant logprob forward.  TEST INFRASTRUCTURE ONLY.

Plain, slow numpy (float32 arithmetic, as the method's statement fixes for the
reference computation) that shares no code with the CUDA library: its own
bf16 / e4m3 codecs, its own norms, attention, top-k, MoE, SSD and log-softmax.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  The product path never calls it and has no CPU
fallback.

Sources (page title, section):

* "Finish RL Training Faster: Bitwise-Consistent, High-Performance,
  Agent-Driven" -- sections "零差异需要一个精确的比较对象" (what must be fixed:
  computation path, quantisation, tie-break, accumulation order),
  "让训练前向使用推理的数值" (batch-invariant GEMM, Top-K tie-break and
  position order, MoE unified rounding, one FP8 KV round trip for every path,
  FP32 fixed-slot expert combine), "一致性有多个层面" (Mamba-2 decode replays the
  prefill chunk order).
* "No More Train-Inference Mismatch: Bitwise Consistent On-Policy
  Reinforcement Learning with vLLM and TorchTitan" -- section "方法细节"
  (fused SiLU MLP and residual + RMSNorm imported into the forward).

The pages print no formulas; every kernel-level definition here is the
plainest reading, listed in the repository's design notes.  Functions whose
result is not pinned by an independent check say "parity unpinned".
"""
