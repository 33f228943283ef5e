// Instantiations of the tiled selective-scan kernel: bf16 inputs, constant-coefficient (per-channel) B and C, the fused scan's input term step * B.
#include "kernel_table.cuh"

namespace ssm {
KernelInfo lookup_bf16_lti(int S, int G, int pass) { return lookup_impl<BF16, true, 0>(S, G, pass); }
}  // namespace ssm
