// gdr_simt.cu -- the CUDA-core path's entry points, and its head sizes K, V in
// {64, 128}; the larger sizes are instantiated in gdr_simt_wide_k.cu (K = 192)
// and gdr_simt_wide_v.cu (V in {192, 256}).  Kernels: gdr_simt_kernels.cuh.
#include "gdr_simt_kernels.cuh"

namespace gdr {

int simt_fwd(const Params &p, int in_f32, int o_f32, int use_cp, cudaStream_t st) {
    if (p.K == 64 && p.V == 64) return fwd_sized<64, 64>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 64 && p.V == 128) return fwd_sized<64, 128>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 128 && p.V == 64) return fwd_sized<128, 64>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 128 && p.V == 128) return fwd_sized<128, 128>(p, in_f32, o_f32, use_cp, st);
    if (p.K == 192) return simt_fwd_wide_k(p, in_f32, o_f32, use_cp, st);
    return simt_fwd_wide_v(p, in_f32, o_f32, use_cp, st);
}

int simt_bwd(const Params &p, int in_f32, int use_cp, cudaStream_t st) {
    if (p.K == 64 && p.V == 64) return bwd_sized<64, 64>(p, in_f32, use_cp, st);
    if (p.K == 64 && p.V == 128) return bwd_sized<64, 128>(p, in_f32, use_cp, st);
    if (p.K == 128 && p.V == 64) return bwd_sized<128, 64>(p, in_f32, use_cp, st);
    if (p.K == 128 && p.V == 128) return bwd_sized<128, 128>(p, in_f32, use_cp, st);
    if (p.K == 192) return simt_bwd_wide_k(p, in_f32, use_cp, st);
    return simt_bwd_wide_v(p, in_f32, use_cp, st);
}

unsigned simt_take_status(cudaStream_t st) {
    return take_status(st) | simt_wide_k_take_status(st) | simt_wide_v_take_status(st);
}

}  // namespace gdr
