// Instantiations of the tiled selective-scan kernel: bf16 inputs, time-varying B and C, the exact zero-order-hold input term.
#include "kernel_table.cuh"

namespace ssm {
KernelInfo lookup_bf16_tv_zoh(int S, int G, int pass) { return lookup_impl<BF16, false, 1>(S, G, pass); }
}  // namespace ssm
