// Kernel instantiations: GBFFT_DEF_COLS_SLAB(7) GBFFT_DEF_COLS_SLAB(8).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_COLS_SLAB(7)
GBFFT_DEF_COLS_SLAB(8)
