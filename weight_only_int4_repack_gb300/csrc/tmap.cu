// Tensor-map (TMA descriptor) encoding with a per-process cache.
//
// A call's tensor maps depend only on the buffer address, its shape and the
// box the kernel copies, so they are encoded once and reused: repeated calls on
// the same buffers (the common case: weights and activation buffers reused
// every step) cost a hash lookup instead of a driver call.
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "w4a16_internal.h"

namespace w4a16 {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

using Key = std::tuple<uintptr_t, int, int, uint64_t, uint64_t, uint64_t, uint64_t, uint64_t, uint32_t, uint32_t,
                       uint32_t, int>;

}  // namespace

bool encode_tmap(CUtensorMap *out, const TmapDesc &d) {
    const Key key{(uintptr_t)d.ptr, d.dtype, d.rank, d.dims[0], d.dims[1], d.dims[2], d.strides[0], d.strides[1],
                  d.box[0], d.box[1], d.box[2], d.swizzle128};
    static std::mutex mu;
    static std::map<Key, CUtensorMap> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *out = it->second;
            return true;
        }
    }
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    for (int i = 0; i < d.rank; ++i) {
        dims[i] = d.dims[i];
        box[i] = d.box[i];
        if (i + 1 < d.rank) strides[i] = d.strides[i];
    }
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map));
    const CUresult r = fn(&map, (CUtensorMapDataType)d.dtype, (cuuint32_t)d.rank, const_cast<void *>(d.ptr), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          d.swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() >= 4096) cache.clear();  // bounded: buffers come and go
    cache[key] = map;
    *out = map;
    return true;
}

bool tmap_weights(CUtensorMap *out, const uint8_t *q_rep, int N, int K, int kblocks_box, int subtiles_box) {
    TmapDesc d{};
    d.ptr = q_rep;
    d.dtype = CU_TENSOR_MAP_DATA_TYPE_UINT64;
    d.rank = 3;
    d.dims[0] = kSubBytes / 8;           // one 512-byte piece as 64 x 8 bytes
    d.dims[1] = (uint64_t)(K / kKBlock);  // k-blocks of a sub-tile
    d.dims[2] = (uint64_t)(N / kSubRows); // sub-tiles
    d.strides[0] = kSubBytes;
    d.strides[1] = (uint64_t)(K / kKBlock) * kSubBytes;
    d.box[0] = kSubBytes / 8;
    d.box[1] = (uint32_t)kblocks_box;
    d.box[2] = (uint32_t)subtiles_box;
    d.swizzle128 = 0;
    return encode_tmap(out, d);
}

bool tmap_activations(CUtensorMap *out, const __half *A, int M, int K, int rows_box) {
    TmapDesc d{};
    d.ptr = A;
    d.dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    d.rank = 2;
    d.dims[0] = (uint64_t)K;
    d.dims[1] = (uint64_t)M;
    d.strides[0] = (uint64_t)K * 2;
    d.box[0] = kKBlock;               // 64 fp16 = one 128-byte swizzle row
    d.box[1] = (uint32_t)rows_box;
    d.swizzle128 = 1;
    return encode_tmap(out, d);
}

bool tmap_activations_kblocks(CUtensorMap *out, const __half *A, int M, int K, int rows_box, int kblocks_box) {
    TmapDesc d{};
    d.ptr = A;
    d.dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    d.rank = 3;
    d.dims[0] = kKBlock;               // 64 k of one k-block (one 128-byte swizzle row)
    d.dims[1] = (uint64_t)M;           // tokens
    d.dims[2] = (uint64_t)(K / kKBlock);  // k-blocks
    d.strides[0] = (uint64_t)K * 2;    // next token
    d.strides[1] = (uint64_t)kKBlock * 2;  // next k-block
    d.box[0] = kKBlock;
    d.box[1] = (uint32_t)rows_box;
    d.box[2] = (uint32_t)kblocks_box;
    d.swizzle128 = 1;
    return encode_tmap(out, d);
}

}  // namespace w4a16
