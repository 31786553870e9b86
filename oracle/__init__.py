"""CPU oracle for mixed-format (FP8 / TQ3) paged decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.  It shares no code, table or constant generator
with the CUDA library; both sides implement the format independently from
the written spec (``include/mkv.h``, section "Storage formats").

What it follows
---------------
The method is the one described in "Minima-KV: Retention-Preserving KV Cache
Compression with Mixed-Format Paged Attention" (arXiv 2608.23834; abstract on
the mlsanity.com paper page, restated on the setupai.cc and aitobox.com
summaries):

* Recent and Anchor pages are kept in FP8, older non-anchor (Stale) pages in a
  packed 3-bit "TQ3" format; every live page stays addressable.
* Format-specific kernels produce partial attention states that a globally
  normalised online-softmax merge combines, with no dense shadow copy.

The pages do not define TQ3 or the FP8 variant; the readings taken here are
listed in the module docstrings and in the header ``include/mkv.h``.

Precision: fp64 throughout, except where floating point decides an integer
code and the spec fixes the precision of that decision (the FP8 quantiser
divides in IEEE fp32, exactly as specified for the library).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force, textbook values or library routines; none
is "parity unpinned" except the pages' own compression ratios (see
``oracle.accounting``).
"""
