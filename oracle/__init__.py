"""Oracle for the ring-attention forward path: plain, slow, fp64, CPU-only.

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg (and its `--impl reference` arm) may import anything from this
package. The product path (online_softmax_merge_gb300 and its CUDA library)
never imports, links or runs it, and this package imports nothing from the
product path. The two share only the seeded input generators, which live in
online_softmax_merge_gb300/inputs.py and hold none of the method's arithmetic.

Sources (web pages on Ring Attention and its online-softmax merge), cited in
each function by page title and section:
  * "Ring Attention" (aarnphm.xyz, thoughts/ring-attention): the ring
    recurrence display that defines S, m, z, y and O = y / z, with the shard
    index b(u, s) = (u - s) mod p.
  * "Ring Attention: Distributed Attention Across Devices" (aicomputerinstitute
    chapter): "Building block: the online-softmax trick" and "Worked example:
    tracing the ring by hand".
  * "Part 4: Ring Attention" (Fofadiya, Illustrated Guide to LLM Inference at
    Scale): sections 4.3 (step-by-step ring), 4.4 (online softmax across KV
    blocks), 4.8.1 (skipping fully-masked blocks).
  * "Ring Attention: what the near-infinite context paper actually says"
    (ashwanijha.dev): "The ring mechanism, step by step", "What the online
    softmax accumulation actually does across rounds", "The causal masking
    complication".
  * Transformer Math "Ring Attention" (aicassindra.com): "The mechanism,
    compressed", "The ring is a prefill algorithm" (the rescale-and-add
    merge of P partial states) and "The backward pass costs a second ring".

Modules:
  attention  dense softmax attention, the plain definition (+ sampled rows)
  ring       the ring recurrence over P virtual shards, fold by fold
  merge      merge of normalised partials (O_p, LSE_p) and finalize (m, z, y)
  shardmap   shard ownership maps, causal visibility, tile classes (brute force)
  backward   dQ, dK, dV of softmax attention (chain rule) and the backward ring

Every function here is pinned by tests under tests/ (test_oracle_*.py) against
values the pages print, closed forms, library routines for special cases,
invariants and brute force on tiny inputs. No function is "parity unpinned".
"""

from . import attention, ring, merge, shardmap, backward  # noqa: F401
