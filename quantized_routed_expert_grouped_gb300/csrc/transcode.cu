// transcode.cu - load-time transcoding of CB2/CB3 weight blobs into the slot layouts CB3X / CB2X.
//
// The idea is that of #3455 "GP100 (sm_60): 4-bit slots for resident IQ2_S / IQ3_XXS / IQ3_S
// gate/up experts", "Problem and result" / "Approach": once the weights are resident, re-encode
// the codebook formats into a layout the decode kernels read without lookups, holding the same
// values so every dot product is unchanged. Here each weight's signed odd value v = +-grid is
// stored as u = (v - 1)/2 + bias (4 bits, bias 8, for CB3X; 2 bits, bias 2, for CB2X), and the
// super-block scale D and the sub-scale nibbles are copied into an 8-byte record per 256 weights.
// One thread per (blob, row, 256-weight chunk); a value that does not fit sets MOE_ERR_CODEBOOK.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) transcode_kernel(int src_type, const int8_t* __restrict__ cb, int dst_type,
                                                        int K, int rows, int n_blobs, const void* const* src_blobs,
                                                        void* const* dst_blobs, int32_t* err) {
    const int nch = K / 256;
    const long long total = static_cast<long long>(n_blobs) * rows * nch;
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int c = static_cast<int>(i % nch);
    const int r = static_cast<int>((i / nch) % rows);
    const int b = static_cast<int>(i / (static_cast<long long>(nch) * rows));
    const bool cb3 = src_type == MOE_CB3;
    const int src_chunk = cb3 ? 102 : 70;
    const int code_bytes = dst_type == MOE_CB3X ? 128 : 64;
    const int bias = dst_type == MOE_CB3X ? 8 : 2, umax = dst_type == MOE_CB3X ? 15 : 3;
    const uint8_t* sb = static_cast<const uint8_t*>(src_blobs[b]) + static_cast<size_t>(r) * nch * src_chunk +
                        static_cast<size_t>(c) * src_chunk;
    uint8_t* drow = static_cast<uint8_t*>(dst_blobs[b]) + static_cast<size_t>(r) * nch * (code_bytes + 8);
    uint32_t words[32];  // the chunk's codes (128 or 64 bytes)
    for (int k = 0; k < 32; ++k) words[k] = 0;
    bool bad = false;
    for (int n = 0; n < 256; ++n) {
        int v;
        if (cb3) {
            v = cb[sb[2 + n / 4] * 4 + (n % 4)];
            if ((sb[66 + n / 8] >> (n % 8)) & 1) v = -v;
        } else {
            v = cb[sb[2 + n / 8] * 8 + (n % 8)];
            if ((sb[34 + n / 8] >> (n % 8)) & 1) v = -v;
        }
        int u = ((v - 1) >> 1) + bias;  // v odd: (v - 1) is even, the shift is exact
        if ((v & 1) == 0 || u < 0 || u > umax) {
            bad = true;
            u = 0;
        }
        const int j = n / 32, w = n % 32;
        int byte, shift;
        if (dst_type == MOE_CB3X) {  // sub-block j: byte w (low nibble) or w-16 (high nibble)
            byte = j * 16 + (w & 15);
            shift = w < 16 ? 0 : 4;
        } else {  // sub-block j: byte w%8, bits 2*(w/8)
            byte = j * 8 + (w & 7);
            shift = 2 * (w >> 3);
        }
        words[byte >> 2] |= static_cast<uint32_t>(u) << (8 * (byte & 3) + shift);
    }
    uint32_t* dc = reinterpret_cast<uint32_t*>(drow + static_cast<size_t>(c) * code_bytes);
    for (int k = 0; k < code_bytes / 4; ++k) dc[k] = words[k];
    uint8_t* rec = drow + static_cast<size_t>(nch) * code_bytes + static_cast<size_t>(c) * 8;
    const uint8_t* sub = sb + (cb3 ? 98 : 66);
    rec[0] = sb[0];
    rec[1] = sb[1];
    rec[2] = 0;
    rec[3] = 0;
    for (int k = 0; k < 4; ++k) rec[4 + k] = sub[k];
    if (bad) set_err(err, MOE_ERR_CODEBOOK);
}

cudaError_t launch_transcode_cb(int src_type, const int8_t* codebook, int dst_type, int K, int rows, int n_blobs,
                                const void* const* src_blobs, void* const* dst_blobs, int32_t* err, cudaStream_t s) {
    const long long total = static_cast<long long>(n_blobs) * rows * (K / 256);
    const long long grid = (total + 255) / 256;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_kernel(transcode_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, false, src_type, codebook,
                         dst_type, K, rows, n_blobs, src_blobs, dst_blobs, err);
}

}  // namespace moe
