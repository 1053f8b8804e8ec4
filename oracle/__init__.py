"""Plain CPU oracle for Prof-K exact top-k selection.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU baseline
leg of ``bench.py`` use it.  It shares no code with the CUDA library.

Everything here is deliberately slow and obvious: numpy / pure Python, fp64 for
every floating-point formula, library sorts as the only "clever" step.

Modules
-------
topk       exact top-k by full sort (the definition), an O(N) restatement of the
           same definition for large inputs, and order-key helpers.
philox     Philox4x64-10 counter-based generator (Salmon et al., SC'11) and the
           sampler: the first S values of a keyed Feistel permutation of [0, n)
           cycle-walked into range (numpy definition).
csample    the same sampler in plain C (sampler.c, built with gcc on first use)
           for the Monte-Carlo checks, held equal to the numpy definition.
hypergeom  hypergeometric pmf / cdf / quantile in fp64.
params     parameter rules: the corrected paper's Algorithm 1 (fast t, M), its
           Theorem 4 (exact t*, M*), and the older version's closed forms
           (Lemma 2, Eq 6, Corollary 4, Theorem 5, its Algorithm 1).
profk      the Prof-K pipeline itself (sample, threshold, filter, check, refine,
           redraw, fallback) written step by step, for stage parity and the
           Monte-Carlo checks of Lemma 1 / Propositions 2-3.  Whether a call
           runs the method or an exact selection is passed in (``route``): a
           library's routing rule is its own, not the pages'.

Pins (what ties each function to something other than itself) live in
``tests/test_oracle_*.py``; every function whose header says "parity unpinned"
has no such pin.
"""
