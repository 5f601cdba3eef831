"""Float64 CPU oracle for paged MLA decode.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, obviously-correct
restatement of what the paged MLA decode path computes. Only the test suite,
the smoke check (``__graft_entry__.smoke``) and the CPU-baseline leg of
``bench.py`` may import it. The product path (the CUDA library and its Python
binding) never calls it and shares no code with it.

Sources (web pages the method is described on):

* [K2.6] "How to serve trillions of tokens for trillion-parameter coding
  agents" (Modal). Section "Tensor parallel was the best parallelism strategy
  for maximum interactivity": one KV entry is 576 elements per token per layer;
  section "First, understand the workload": the model has no distinct keys and
  values; section "Use custom speculative decoding ...": the target model
  checks the drafted tokens in parallel without changing its distribution.
* [CF] "Smaller, faster, safer: running Kimi and GLM at scale" (Cloudflare).
  Section "Quantizing the KV cache": the cache is stored as FP8 e4m3 and the
  attention kernel converts values as it reads them. Section "Protecting a
  shared KV cache": many requests read pages of one physical paged cache, and
  a per-page tag that changes on reallocation is checked before decode reads.
* [vLLM] "vLLM x AgentX: Optimizing for Real-World Agentic Serving".
  Section "Kimi K3": MLA keeps one latent head; decode context parallelism
  produces partial attention outputs plus log-sum-exp statistics that are
  merged with online softmax.

Modules:

* :mod:`oracle.e4m3` -- the OCP FP8 E4M3 ("fn") codec: decode table and
  round-to-nearest-even, saturating encode of ``x / kv_scale``.
* :mod:`oracle.attention` -- page gather, dequantisation, causal draft
  visibility, float64 softmax attention, log-sum-exp merge, and a brute-force
  dense path for tiny inputs.
* :mod:`oracle.integrity` -- the KV-cache integrity check of [CF] section
  "Protecting a shared KV cache": per-request comparison of the pages' current
  tags with the tags the request expects, one status word per request.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines, brute force and invariants (see each test's docstring).
"""

from . import attention, e4m3, integrity  # noqa: F401
