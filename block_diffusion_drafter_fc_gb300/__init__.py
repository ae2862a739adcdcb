"""DFlash drafter block step on GB300 (sm_103a): C-ABI library libdflash + binding.

`synth` draws the seeded synthetic workloads; `dflash` loads libdflash.so and
marshals arguments to it (import it explicitly: it fails loudly when the
library is missing).  `build` compiles the library with nvcc.
"""
