// Instantiations of the tiled selective-scan kernel: bf16 inputs, time-varying B and C, the Mamba-block prologue (causal conv of width 4 + silu on x).
#include "kernel_table.cuh"

namespace ssm {
KernelInfo lookup_bf16_tv_conv(int S, int G, int pass) { return lookup_impl<BF16, false, 2>(S, G, pass); }
}  // namespace ssm
