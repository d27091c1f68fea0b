"""CPU oracle for the paged KV cache write and paged attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check
(``__graft_entry__.smoke``) and the benchmark's CPU-baseline leg
(``bench.py``'s ``cpu_baseline`` / ``--impl reference``) may import or call
anything in this package.  The CUDA library never does: it has no CPU
fallback, and this package shares no code, table or helper with it.

The oracle is the plain definition of what the hot path computes, written
in numpy with float64 arithmetic:

* the copy-on-write block copy follows "Build a Mini vLLM", Key Takeaways
  6 (prefix sharing with copy-on-write blocks);
* slot mapping, the scatter write and the block-table gather follow
  "Build a Mini vLLM" section 2 (``BlockManager.append_slot``) and section 3
  (``gather_kv``), and "Day 16" (What I learned, item 3: write is a scatter,
  read is a gather);
* attention follows "Build a Mini vLLM" section 3 (``paged_attention``:
  softmax(q . k / sqrt(d)) . v per query head, GQA heads expanded with
  repeat-interleave) and section 4 (the causal ``triu(1)`` mask of prefill);
* the split-KV partials and their merge are the online-softmax identity,
  which reduces to the same softmax (pages silent; exact in real arithmetic).

Every function is pinned by tests in ``tests/test_oracle_pins.py`` against
values and properties the pages and mathematics fix (worked examples under
``tests/golden/``, closed forms, a library attention routine, invariants).
No function is "parity unpinned".
"""
from .paged import (  # noqa: F401
    to_float64,
    slot_of,
    slot_mapping,
    kv_write,
    copy_blocks,
    gather_kv,
    kv_head_of,
    causal_last_key,
    attend,
    paged_attention_decode,
    paged_attention_prefill,
    partial_attention,
    merge_partials,
    paged_attention_decode_split,
)
