// Paged decode attention: f32 instantiations of the partition and merge kernels.
#include "pa_decode.cuh"

namespace pagedkv {

cudaError_t launch_decode_f32(const DecodeLaunch &L, cudaStream_t stream)
{
    return launch_decode_dispatch<float>(L, stream);
}

int plan_grid_f32(const DecodeLaunch &L) { return plan_grid_dispatch<float>(L); }

size_t decode_smem_bytes_f32(int head_dim, int block_size, int group)
{
    return smem_dispatch<float>(head_dim, block_size, group);
}

}  // namespace pagedkv

PA_TRACE_DEFINE_READER(f32)
