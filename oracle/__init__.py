"""CPU oracle for the selected-token logprob -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import, call, link or execute
anything in this package.  The product path (the CUDA library and its Python
binding) never touches it and fails loudly when its own extension is missing.

Two independent checkers live here, sharing no code with the CUDA path:

* ``linear_logprob`` -- the definition, written out in fp64 with numpy.
* ``contract_emulator.c`` (loaded by ``emulator``) -- the fixed fp32 numeric
  contract (vocab-tile split, in-tile pairwise tree, merge operator, tile
  tree, own exp/log, rounding points) written again in plain C, so that the
  GPU's bits can be predicted exactly from inputs whose logits are exact.
"""
