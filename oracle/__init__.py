"""CPU oracle for the Medusa tree-verify decode step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct float64 (numpy) restatement of what the
method computes, written from the pages' definitions before any GPU kernel.
It shares no code with the CUDA path; the only shared module is ``synth``
(seeded input generators). Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import it. The product path
never calls it.

Sources (cited by page title and section):

* "大模型推理 memory bandwidth bound (5) - Medusa" (dtcms.com): 一.1 Medusa
  heads, 一.2 Tree attention, 一.3 Typical acceptance, 二.2
  generate_medusa_buffers(), 二.3 initialize_medusa(), 二.4
  generate_candidates(), 二.5 tree_decoding(), 二.6 evaluate_posterior(),
  二.7 update_inference_inputs().
* "Phi-3-mini-128k-instruct_rai_1.8.0_medusa_1.0_npu" article (lqnn.cn):
  2️⃣ (greedy output identical to the base model), 4️⃣ (tree attention mask).

Modules: ``tree`` (static tree buffers), ``model`` (Llama-style backbone,
Medusa heads, tree attention), ``posterior`` (greedy and typical acceptance),
``kv`` (KV compaction), ``decode`` (candidates, verify step, greedy loops),
``sampling`` (typical and nucleus one-token root sampling).

Pins (what ties each function to something other than itself) are the
``-m "not gpu"`` tests in ``tests/test_oracle_*.py``. Every function here is
pinned; none is "parity unpinned".
"""
