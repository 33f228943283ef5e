// Instantiations of the tiled selective-scan kernel: f32 inputs, constant-coefficient (per-channel) B and C, the fused scan's input term step * B.
#include "kernel_table.cuh"

namespace ssm {
KernelInfo lookup_f32_lti(int S, int G, int pass) { return lookup_impl<F32, true, 0>(S, G, pass); }
}  // namespace ssm
