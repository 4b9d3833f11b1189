"""CPU oracle for the grouped MXFP8 MoE expert FFN -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy (float64) restatement of what the
hot path computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  The CUDA library shares no code
with it: no kernels, headers, tables or helpers.  Inputs reach it as plain
arrays from the seeded generator; it never reads anything produced by the
CUDA path.

Sources (the pages this follows; citations name the page and its section):

* [BioNeMo-MoE] "Efficient MoE Training for Biological Foundation Models"
  (scopeai.cc summary of the NVIDIA technical blog).  Sections:
  "MoE训练的瓶颈与TE的对应能力" (bottlenecks: per-expert Python loop, 8-bit
  MXFP8 with one scale per 32 consecutive values, 16-bit master weights with
  separate quantize/dequantize steps);
  "GroupedLinear：把逐专家循环改成一次分组GEMM" (one grouped GEMM driven by
  per-expert token counts split_sizes; each expert keeps its own weight;
  gate_up has out_features = 2 * intermediate_size, bias=False);
  "MXFP8与融合MLP：减少显存并跳过独立量化步骤" (gate_up -> ScaledSwiGLU ->
  down, the router probabilities multiply the SwiGLU output; fused forward
  and backward ops).
* [AutoModel] "英伟达开源MoE加速神器：一行代码，微调快3.7倍" (openai-hub.com),
  section "三板斧" (tokens are routed to a few of many experts; the expert
  FFN is the compute bulk; grouped GEMM packs the experts' matmuls).

Modules: ``mxfp8`` (E4M3 codec, power-of-two block scale, block quantizer),
``routing`` (top-k softmax routing, expert-major permutation),
``expert_ffn`` (per-expert loop forward and backward, combine).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
brute force, invariants, finite differences or textbook special cases.
"""
