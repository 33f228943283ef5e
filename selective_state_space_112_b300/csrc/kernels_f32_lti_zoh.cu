// Instantiations of the tiled selective-scan kernel: f32 inputs, constant-coefficient (per-channel) B and C, the exact zero-order-hold input term.
#include "kernel_table.cuh"

namespace ssm {
KernelInfo lookup_f32_lti_zoh(int S, int G, int pass) { return lookup_impl<F32, true, 1>(S, G, pass); }
}  // namespace ssm
