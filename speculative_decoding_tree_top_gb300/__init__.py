"""DominoTree drafting-round tree builder for GB300 (sm_103a): top-M candidate selection and the conditional
best-first draft-tree builder, as hand-written CUDA behind a C ABI (include/dominotree.h)."""
