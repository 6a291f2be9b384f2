// Kernel instantiations: GBFFT_DEF_RPAIR(13..14).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_RPAIR(13)
GBFFT_DEF_RPAIR(14)
