// Device-side reorder of integer weight codes into the GEMM's compute order
// (the packed format documented in qoq_internal.h), and its inverse for tests.
// The idea follows the compute-aware weight reordering of "QServe: W4A8KV4
// Quantization and System Co-design for Efficient LLM Serving" (papercache
// summary, section "计算感知权重重排序"; zenmind review 3.2): weights are static,
// so they are stored once in the exact order the main loop consumes them.
// Here that order is one 8 KB block per (128-row tile, 128-k group), copied
// whole by one bulk TMA, laid out so that each converter thread reads 16-byte
// chunks without shared-memory bank conflicts.
#include "qoq_internal.h"

namespace qoq {
namespace {

// grid: (K/128, N/128); 512 threads, one 16-byte code chunk each.
__global__ void pack_kernel(const uint8_t *__restrict__ q4, const uint8_t *__restrict__ s_g,
                            const uint8_t *__restrict__ zp, int N, int K, int group,
                            uint8_t *__restrict__ packed) {
    const int kg = blockIdx.x, nt = blockIdx.y;
    const int G = K / kTileK;
    const int c = threadIdx.x, p = c >> 7, r = c & 127;
    const int n = nt * kTileN + r;
    const uint32_t bb = block_bytes(group);
    uint8_t *blk = packed + kHeaderBytes + (static_cast<size_t>(nt) * G + kg) * bb;
    PackedHeader *hdr = reinterpret_cast<PackedHeader *>(packed);

    int s = 1, z = 0;
    if (group) {
        s = s_g[static_cast<size_t>(n) * G + kg];
        z = zp[static_cast<size_t>(n) * G + kg];
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(q4 + static_cast<size_t>(n) * K + kg * kTileK + 32 * p);
    uint4 a = src[0], b = src[1];
    const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t illegal = 0;
    uint32_t out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w = 0;
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
            const int k_lo = 8 * j + bi, k_hi = k_lo + 4;
            const uint32_t clo = (in[k_lo >> 2] >> ((k_lo & 3) * 8)) & 0xffu;
            const uint32_t chi = (in[k_hi >> 2] >> ((k_hi & 3) * 8)) & 0xffu;
            illegal += (clo > 15u) + (chi > 15u);
            if (group) {
                const int wl = (static_cast<int>(clo) - z) * s, wh = (static_cast<int>(chi) - z) * s;
                illegal += (wl < -128 || wl > 127) + (wh < -128 || wh > 127);
            }
            w |= ((clo & 15u) | ((chi & 15u) << 4)) << (8 * bi);
        }
        out[j] = w;
    }
    reinterpret_cast<uint4 *>(blk)[c] = make_uint4(out[0], out[1], out[2], out[3]);

    if (c < 128) {
        if (group) {
            illegal += (s > 17) + (z > 15);
            // sum of the row's 128 codes in this group (used by the fp8 path)
            const uint4 *row = reinterpret_cast<const uint4 *>(q4 + static_cast<size_t>(n) * K + kg * kTileK);
            uint32_t sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = row[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    sum += ((w[j] & 0xffu) + ((w[j] >> 8) & 0xffu) + ((w[j] >> 16) & 0xffu) + (w[j] >> 24)) & 0xffffu;
            }
            blk[kCodeBytes + 4 * r] = static_cast<uint8_t>(s);
            blk[kCodeBytes + 4 * r + 1] = static_cast<uint8_t>(z);
            blk[kCodeBytes + 4 * r + 2] = static_cast<uint8_t>(sum & 0xffu);
            blk[kCodeBytes + 4 * r + 3] = static_cast<uint8_t>(sum >> 8);
        } else if (kg == 0) {
            const int zc = zp[n];
            illegal += (zc > 15);
            packed[packed_z_offset(N, K) + n] = static_cast<uint8_t>(zc);
        }
    }
    if (illegal) atomicAdd(&hdr->illegal, illegal);
    if (kg == 0 && nt == 0 && c == 0) {
        hdr->magic = kPackedMagic;
        hdr->version = kPackedVersion;
        hdr->N = N;
        hdr->K = K;
        hdr->group = group;
        hdr->block_bytes = bb;
    }
}

__global__ void unpack_kernel(const uint8_t *__restrict__ packed, int N, int K, int group,
                              uint8_t *__restrict__ q4, uint8_t *__restrict__ s_g,
                              uint8_t *__restrict__ zp) {
    const int kg = blockIdx.x, nt = blockIdx.y;
    const int G = K / kTileK;
    const int c = threadIdx.x, p = c >> 7, r = c & 127;
    const int n = nt * kTileN + r;
    const uint32_t bb = block_bytes(group);
    const uint8_t *blk = packed + kHeaderBytes + (static_cast<size_t>(nt) * G + kg) * bb;
    const uint4 v = reinterpret_cast<const uint4 *>(blk)[c];
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
            const uint32_t byte = (in[j] >> (8 * bi)) & 0xffu;
            const int k_lo = 8 * j + bi, k_hi = k_lo + 4;
            out[k_lo >> 2] |= (byte & 15u) << ((k_lo & 3) * 8);
            out[k_hi >> 2] |= (byte >> 4) << ((k_hi & 3) * 8);
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(q4 + static_cast<size_t>(n) * K + kg * kTileK + 32 * p);
    dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
    dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    if (c < 128) {
        if (group) {
            s_g[static_cast<size_t>(n) * G + kg] = blk[kCodeBytes + 4 * r];
            zp[static_cast<size_t>(n) * G + kg] = blk[kCodeBytes + 4 * r + 1];
        } else if (kg == 0) {
            zp[n] = packed[packed_z_offset(N, K) + n];
        }
    }
}

}  // namespace

cudaError_t launch_pack(const uint8_t *q4, const uint8_t *s_g, const uint8_t *z, int N, int K,
                        int group, void *packed, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(packed, 0, kHeaderBytes, stream);
    if (e != cudaSuccess) return e;
    dim3 grid(K / kTileK, N / kTileN);
    pack_kernel<<<grid, 512, 0, stream>>>(q4, s_g, z, N, K, group, static_cast<uint8_t *>(packed));
    return cudaGetLastError();
}

cudaError_t launch_unpack(const void *packed, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                          uint8_t *z, cudaStream_t stream) {
    dim3 grid(K / kTileK, N / kTileN);
    unpack_kernel<<<grid, 512, 0, stream>>>(static_cast<const uint8_t *>(packed), N, K, group, q4,
                                            s_g, z);
    return cudaGetLastError();
}

}  // namespace qoq
