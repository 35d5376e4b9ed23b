"""CPU oracle for paged decode / step attention -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the pages define, used
only by ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py``.  The CUDA library never imports,
links or calls anything here, and nothing here imports the library.

Precision: float64 throughout, except where the pages fix float32 (the RoPE
frequency table and the angle product, "Phi-3 Mini 4K Instruct -- files",
src/rope.linnet, ``tables``).  Tensors are bf16 bit patterns (uint16).

Modules
  bf16   -- bf16 <-> float64 conversion (round to nearest even from float64)
  rope   -- frequency tables (plain theta, llama3 three-band rescale), rotation,
            per-head QK-norm
  paged  -- slot placement, append (rope + write), visible key range, attention
            over a row's pages (decode rows and packed prompt chunks), and the
            row-based packed-prompt rule used to cross-check the chunk path

Every function is pinned by ``tests/test_oracle_pins.py`` against facts the
pages or the mathematics fix; ``tests/test_oracle_mutations.py`` plants
plausible mistakes in these modules and checks that a pin catches each one.
"""
from . import bf16, rope, paged  # noqa: F401
