// Kernel instantiations: GBFFT_DEF_COLS_TW(11).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_COLS_TW(11)
