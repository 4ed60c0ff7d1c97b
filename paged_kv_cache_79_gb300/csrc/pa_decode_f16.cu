// Paged decode attention: f16 instantiations of the partition and merge kernels.
#include "pa_decode.cuh"

namespace pagedkv {

cudaError_t launch_decode_f16(const DecodeLaunch &L, cudaStream_t stream)
{
    return launch_decode_dispatch<__half>(L, stream);
}

int plan_grid_f16(const DecodeLaunch &L) { return plan_grid_dispatch<__half>(L); }

size_t decode_smem_bytes_f16(int head_dim, int block_size, int group)
{
    return smem_dispatch<__half>(head_dim, block_size, group);
}

}  // namespace pagedkv

PA_TRACE_DEFINE_READER(f16)
