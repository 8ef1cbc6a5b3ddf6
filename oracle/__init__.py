"""fp64 CPU oracle for the hybrid Muon + AdamW optimizer step.

TEST INFRASTRUCTURE ONLY. Nothing in the product (the ``adamw_hybrid_optimizer_gb300``
package and its CUDA library) imports, links or runs anything here. Only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it.

It is a plain, slow, obviously correct restatement of what the web pages describe,
written from their formulas and prose in float64 NumPy:

  oracle.muon          Muon: momentum, Nesterov input, Frobenius normalisation,
                       transpose-to-wide, quintic Newton-Schulz, 0.2*sqrt(max(A,B))
                       scaling, decoupled (optionally cautious) weight decay; and the
                       same iteration run in the m x m Gram space (newton_schulz_gram).
  oracle.adamw         AdamW with bias correction and decoupled decay; Adam + L2.
  oracle.buckets       grouping of Muon matrices by shape into (K, A, B) stacks.
  oracle.polar_express per-step minimax odd-quintic coefficients (Polar Express).
  oracle.bf16          round-to-nearest-even to bfloat16, for stored outputs.

Sources (web pages, cited by title and section):
  [P1] "MuonAdamW vs DistMuonAdamW: Key Differences for Single and Multi-GPU Training
       in nanochat" (instagit.com)
  [P2] "Optimizers: AdamW, Muon and the distributed optimizer" (AI-infra handbook,
       anrans.github.io)
  [P3] "dtensor-muon 0.1.0" package description (PyPI)
  [P4] "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead" (gist.science
       summary of arXiv 2606.27153)

Every function is pinned by ``tests/test_oracle_*.py`` against something other than
itself (SVD closed forms, the pages' printed worked examples, torch.optim's AdamW and
Adam, brute force), except the fidelity of the Polar Express table to the published
paper, which no page prints: parity unpinned for that table's *values* (the solver
that produces them is pinned by the equioscillation theorem and a closed form).
"""
