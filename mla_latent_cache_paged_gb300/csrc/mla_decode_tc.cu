// Tensor-core (tcgen05/TMEM + TMA) decode kernel: not built yet.
#include "mla_internal.h"

namespace mla {

bool tc_kernel_built() { return false; }

int launch_decode_tc(const DecodeParams&, int, void*) { return 1; }

}  // namespace mla
