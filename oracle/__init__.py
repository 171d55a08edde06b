"""Oracle for the Muon owner step: a plain, slow, obviously correct CPU
restatement in float64 (NumPy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library under
``matrix_optimizers_gb300/`` never imports it, links it or shares code with it;
the two meet only on inputs drawn by ``workloads/`` (which holds no arithmetic
of the method).

What each module restates, and from where:

* ``muon``    -- heavy-ball momentum, Frobenius normalisation, the m<=n
                 orientation, the quintic Newton-Schulz (NS) iteration and the
                 scaled weight update.  The pages ("Riepilogo Tecnico: SignMuon",
                 §2 "Meccanismo Principale" item 1 and "Flusso Algoritmico"
                 step 1; "Riassunto Tecnico: MatrixFSDP", §Metodologia 1) say the
                 owner runs Muon's NS orthogonalisation of the momentum locally;
                 they do not print the polynomial, so the standard Muon quintic
                 X <- aX + b(XX^T)X + c(XX^T)^2 X with (a,b,c) =
                 (3.4445, -4.7750, 2.0315), k = 5, X0 = M/||M||_F is used.
* ``sign``    -- Sign-Muon sign extraction, 1-bit packing, majority vote and
                 the voted update (SignMuon §2 "Flusso Algoritmico" steps 2-4,
                 "Meccanismo Principale" item 3).
* ``adamw``   -- decoupled AdamW for the 1D tail (MatrixFSDP §Metodologia 1,
                 "Tensori Non-Matriciali").
* ``planner`` -- the owner planner balancing resident bytes and optimizer work
                 (MatrixFSDP §Metodologia 2, "Metadati MatrixShard & Global
                 Planner"), read as longest-processing-time greedy.
* ``bf16``    -- round-to-nearest-even to bfloat16, for state the method stores
                 in bf16.

Pins (tests/test_oracle_*.py): SVD closed form of NS, the polar factor reached
by the cubic NS special case, scale / transpose / orthogonal invariances,
brute-force sign voting over every sign pattern, the t=1 closed form of AdamW
and torch.optim.AdamW, exact LPT results derived by hand, brute-force optimal
schedules.  Every function here has at least one such pin.
"""
