"""CPU oracle for the DFlash2 block-parallel draft step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or execute anything in this package.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline and
reference legs of ``bench.py`` use it.  It shares no code with the CUDA path.

The oracle is plain numpy in float64.  Each function cites the passage of
the source pages it follows, by page title and section:

* [NIM]      "DFlash2 Speculative Decoding | NVIDIA NIM for Alpamayo
              Documentation" (sections "Observe Acceptance",
              "Bring Your Own DFlash2 Head").
* [vLLM]     "DFlash speculative decoding with vLLM" (sections
              "Requirements", "DFlash2 inference", "Validation").
* [llama]    "DFlash2 Speculative Decoding" (llama-cpp-python wiki;
              sections "Goal", "Prerequisites", "Compare With Ordinary
              Decoding", "Configuration Notes").
* [Train]    "Train a DFlash Drafter for Speculative Decoding" (sections
              "What is DFlash?", "Variants", "Objective", "Data",
              "Key Config Fields").

Where the pages leave a step open, the docstring says which reading was
taken ("Reading taken: ...").  Functions whose result
cannot be pinned to anything but their own definition say "parity unpinned".
"""

from .dflash2_oracle import *  # noqa: F401,F403
