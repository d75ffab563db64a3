"""CPU oracle for the ReplaySSM decode hot path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 implementations of what the decode path must compute,
written from the pages' descriptions:

* ``recurrence``  the conventional per-token Mamba-2 and Gated DeltaNet
  recurrences (state read, rank-1 update, output), which ReplaySSM must
  reproduce up to floating-point rounding.
* ``ring``        the ring-buffer cursor (head, count) with flush on fill,
  pointer-advance commit and explicit flush, as plain integers.
* ``layer``       the expected results of every C-ABI call (decode step,
  verify, commit, flush) on any subset of sequences.
* ``codecs``      e4m3 / e2m1 encoders and decoders and the two read-copy
  formats (FP8 per-row scale, NVFP4 16-element blocks).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it, and
it shares no code with the CUDA library; both take inputs from the seeded
generators in ``workloads``.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, invariants and brute-force exact cases from the pages'
mathematics (see each function's docstring for the passage followed).
Sources are cited by page title and section:

* [richland] "ReplaySSM caches SSM inputs instead of state, cutting
  hybrid-model decode traffic in half" (richland.au), sections
  "What shipped", "Why it matters", "Caveats".
* [ai-jitan] "NVIDIAとプリンストン大Dao AI Lab、ハイブリッドモデルの推論を速める
  「ReplaySSM（リプレイSSM）」を公開" (ai-jitan-hub.com), sections
  "ReplaySSMは何をする手法か", "何がどれだけ速くなったのか" (items 1-3).
* [warp-studio] "ReplaySSM：ハイブリッドモデルの高速デコーディングを実現する
  状態ストレージ再考" (ai.warp-studio.com), sections
  "ReplaySSMによる高速化メカニズムと性能ベンチマーク",
  "推測デコーディングにおける革新と実装詳細".
"""
