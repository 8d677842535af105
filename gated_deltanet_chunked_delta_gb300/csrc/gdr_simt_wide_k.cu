// gdr_simt_wide_k.cu -- the CUDA-core path at K = 192 (V in {64, 128, 192,
// 256}).  Kernels: gdr_simt_kernels.cuh.
#include "gdr_simt_kernels.cuh"

namespace gdr {

int simt_fwd_wide_k(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st) {
    switch (p.V) {
        case 64: return fwd_sized<192, 64>(p, in_f32, o_f32, use_cp, st);
        case 128: return fwd_sized<192, 128>(p, in_f32, o_f32, use_cp, st);
        case 192: return fwd_sized<192, 192>(p, in_f32, o_f32, use_cp, st);
        case 256: return fwd_sized<192, 256>(p, in_f32, o_f32, use_cp, st);
    }
    return 1;
}

int simt_bwd_wide_k(const Params &p, int in_f32, int use_cp, cudaStream_t st) {
    switch (p.V) {
        case 64: return bwd_sized<192, 64>(p, in_f32, use_cp, st);
        case 128: return bwd_sized<192, 128>(p, in_f32, use_cp, st);
        case 192: return bwd_sized<192, 192>(p, in_f32, use_cp, st);
        case 256: return bwd_sized<192, 256>(p, in_f32, use_cp, st);
    }
    return 1;
}

unsigned simt_wide_k_take_status(cudaStream_t st) { return take_status(st); }

}  // namespace gdr
