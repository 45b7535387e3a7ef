// rs_sort_u32.cu -- instantiates the sort kernels and driver for one key type
// (kept in its own translation unit so the key types compile in parallel).
#include "rs_kernels.cuh"

namespace rs {
template rs_status run_sort<KU32>(Plan& pl);
}  // namespace rs
