"""fp64 CPU oracle for the SnapKV / H2O / StreamingLLM KV-cache hot path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg (``cpu_baseline`` and ``--impl reference``) may
import or call anything in this package.  The CUDA library never routes through it,
and it shares no code, header, table or helper with
``attention_score_kv_snapkv_gb300/``: neither side imports the other.  The only
code both sides see is the seeded input generator in ``workloads/``, which holds
none of the method's arithmetic.

Everything here is plain numpy in float64, written step by step in the order the
articles describe the methods, without blocking, fusion or reordering:

* ``oracle.attention`` -- softmax attention of one query over a set of keys
  (the "All KV" full-cache baseline that the SnapKV and H2O articles compare with).
* ``oracle.snapkv``    -- SnapKV: window scoring, vote, 1D max-pool, per-head top-k,
  gather of the compact cache (SnapKV article, section 処理の流れ "processing flow",
  steps 1-4; section 推論方法 "inference").
* ``oracle.h2o``       -- H2O: cumulative attention score, heavy-hitter + recent-window
  eviction (H2O article, sections 何を残すのか "what is kept" and 処理の流れ).
* ``oracle.streaming`` -- StreamingLLM: sink tokens plus a recent ring buffer
  (StreamingLLM article, sections キャッシュ構造 "cache structure" and 推論の流れ
  "inference flow").

Pins: every function is checked by ``tests/test_oracle_*.py`` against closed forms,
invariants, hand-worked examples (``tests/golden/``) and brute force on tiny inputs.
Model-quality claims of the articles (needle retrieval, LongBench, perplexity) need
trained weights and datasets and are parity unpinned; they are not computed here.
"""

from . import attention, h2o, snapkv, streaming  # noqa: F401
