"""Float64 CPU oracle for mixed-fidelity paged KV attention, gather and demotion.

TEST INFRASTRUCTURE ONLY. Nothing in the product path (the ``ekv`` CUDA library and
its Python binding) imports, links or executes anything in this package. Only the
tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs
of ``bench.py`` may use it.

It is written from the pages' statement of the problem, plainly and slowly:

* ``e4m3``   -- the OCP OFP8 E4M3 ("FN") value set and round-to-nearest-even,
                saturating encoder (pages name E4M3 only: knlp.io "Asymmetric K16/V8
                KV cache", Fig. "Fresh prefill gets a fast path"; DPS paper Sec. 2).
* ``decode`` -- paged GQA decode attention over dequantised pages (ElasticKV Sec. 2.1
                paged block table, Sec. 3.2 dual-mode attention; knlp.io decode prefix
                "reads persistent FP16 keys and FP8 values", scales "still apply in
                attention").
* ``gather`` -- compact-prefill gather of K16/V8 pages into an FP16 workspace
                (knlp.io "What changes in vLLM's prefill routing?").
* ``base``   -- ElasticKV BASE value pages (FP16 high byte, low byte zero-filled):
                value, TARGET -> BASE demotion, exact promotion (ElasticKV Sec. 3.2,
                App. B.2-B.3).
* ``elastic`` -- ElasticKV's pair-structured value layout (value locations as half
                slots, a separate value block table), TARGET-BASE-TARGET boundaries, the
                batch-level BASE indicator and located transitions (Sec. 3.1-3.2, App. B).
* ``prefill`` -- FP16 causal prefill of whole prompts over the gathered workspace
                 (knlp.io "What changes in vLLM's prefill routing?": native FP16 prefill).
* ``writer`` -- the K16/V8 cache writer: one new token per sequence into its page row
                (knlp.io implementation checks: "K bit-exact, V within FP8 noise").
* ``demote`` -- TARGET -> compact requantisation of FP16 value pages with absmax
                scales (ElasticKV Sec. 3.4 "Transition protocols", with the compact
                format of the knlp.io page).

Every function computes in float64 (or exactly, for the integer/byte work) and shares
no code with the CUDA path. Pins that tie each function to something other than
itself live in ``tests/test_oracle_*.py``.
"""

from . import base, e4m3, decode, gather, demote, writer, elastic, prefill  # noqa: F401

PAGE_SIZE = 16
MODE_TARGET_FP16 = 0
MODE_COMPACT_E4M3 = 1
SCALE_PER_TENSOR = 0
SCALE_PER_PAGE_HEAD = 1
