// tcgen05 split-KV chunk kernel: tensor-map encoding and the variant table.
#include <cudaTypedefs.h>

#include <atomic>

#include "params.h"

namespace kvd {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

}  // namespace

bool tc_encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, bool u8) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

const ChunkKernel* tc_table_d64(bool f32, int qr);
const ChunkKernel* tc_table_d128(bool f32, int qr);
const ChunkKernel* tc_table_d256(bool f32, int qr);
const ChunkKernel* tc8_table_d128(bool f32, int qr, bool fp8);
const ChunkKernel* tc8_table_d256(bool f32, bool fp8);

// Q is stored in blocks of the group size rounded up (48 or 64 rows: groups
// of up to 48 leave room for a third K stage at head_dim 256); several query
// tokens whose rows (T times the group rounded up to 8) fit in 128 run on the
// 128-row variant, which stacks them in one tile.
const ChunkKernel* tc_chunk_kernel(int head_dim, bool f32_out, int group, int T) {
    if (group < 17 || group > 64 || T < 1) return nullptr;
    const int qr = (T > 1 && T * ((group + 7) & ~7) <= 128) ? 128 : (group <= 48 ? 48 : 64);
    switch (head_dim) {
        case 64: return tc_table_d64(f32_out, qr);
        case 128: return tc_table_d128(f32_out, qr);
        case 256: return tc_table_d256(f32_out, qr);
        default: return nullptr;
    }
}

// 8-bit caches (contiguous or paged) with groups of 17..64 (head_dim 128) or 17..48
// (head_dim 256, where a 64-row Q block leaves no room for two 8-bit stages
// per tensor): the converting variant, one query token per tile (several run
// as virtual sequences).
const ChunkKernel* tc8_chunk_kernel(int head_dim, bool f32_out, int group, bool fp8) {
    if (group < 17 || group > 64) return nullptr;
    if (head_dim == 128) return tc8_table_d128(f32_out, group <= 48 ? 48 : 64, fp8);
    if (head_dim == 256 && group <= 48) return tc8_table_d256(f32_out, fp8);
    return nullptr;
}

}  // namespace kvd
