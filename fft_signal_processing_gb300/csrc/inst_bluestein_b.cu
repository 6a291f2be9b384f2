// Kernel instantiations: GBFFT_DEF_BLUESTEIN(11) GBFFT_DEF_BLUESTEIN(12).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_BLUESTEIN(11)
GBFFT_DEF_BLUESTEIN(12)
