// Sharded checkpoint files: one file per rank holding that rank's shard of the
// fp32 master weights and Adam moments (and optionally its bf16 weights), with
// a header that records the layout and a CRC-32 of the payload.
//
// "ZeRO Optimizer, in depth", "Checkpoints: sharded on the way in, consolidated
// on the way out": every rank writes its own shard of model and optimizer
// state plus a small metadata file, so saving needs no gather; a consolidation
// step rebuilds a plain full-precision state for a different layout.
//
// Host-only code: the caller copies device shards to host memory first.  The
// CRC is the reflected CRC-32 of IEEE 802.3 (polynomial 0xEDB88320, initial
// value and final xor 0xFFFFFFFF), computed eight bytes at a time with eight
// 256-entry tables built on first use ("slicing by 8": table k maps a byte to
// its CRC contribution k bytes further on; the bytes are read little-endian,
// the byte order of x86-64 and AArch64 hosts alike).
#include <cstdio>
#include <cstring>
#include <mutex>

#include "zero_gb300.h"

namespace {

constexpr char kMagic[8] = {'Z', 'G', 'B', 'S', 'H', 'A', 'R', 'D'};
constexpr uint32_t kVersion = 1;
// The library's element limit (that of zero_layout): every byte count below fits.
constexpr int64_t kMaxShardElems = INT64_MAX / 8;

uint32_t g_crc_table[8][256];
std::once_flag g_crc_once;

void build_crc_table() {
    for (uint32_t i = 0; i < 256; ++i) {
        uint32_t c = i;
        for (int k = 0; k < 8; ++k) c = (c & 1u) ? (0xEDB88320u ^ (c >> 1)) : (c >> 1);
        g_crc_table[0][i] = c;
    }
    for (int t = 1; t < 8; ++t)
        for (uint32_t i = 0; i < 256; ++i) {
            const uint32_t c = g_crc_table[t - 1][i];
            g_crc_table[t][i] = (c >> 8) ^ g_crc_table[0][c & 0xffu];
        }
}

uint32_t load_le32(const unsigned char* p) {
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

uint32_t crc_update(uint32_t crc, const void* data, size_t n) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    const uint32_t(&T)[8][256] = g_crc_table;
    for (; n >= 8; n -= 8, p += 8) {
        const uint32_t lo = crc ^ load_le32(p);
        const uint32_t hi = load_le32(p + 4);
        crc = T[7][lo & 0xffu] ^ T[6][(lo >> 8) & 0xffu] ^ T[5][(lo >> 16) & 0xffu] ^ T[4][lo >> 24] ^
              T[3][hi & 0xffu] ^ T[2][(hi >> 8) & 0xffu] ^ T[1][(hi >> 16) & 0xffu] ^ T[0][hi >> 24];
    }
    for (; n > 0; --n, ++p) crc = T[0][(crc ^ *p) & 0xffu] ^ (crc >> 8);
    return crc;
}

struct FileHeader {
    char magic[8];
    uint32_t version;
    uint32_t flags;          // bit 0: bf16 weights present
    zero_ckpt_header_t h;
    uint32_t crc;            // CRC-32 of the payload
    uint32_t reserved;
};

bool write_all(FILE* f, const void* p, size_t n) {
    return n == 0 || std::fwrite(p, 1, n, f) == n;
}

bool read_all(FILE* f, void* p, size_t n, uint32_t* crc) {
    if (n == 0) return true;
    if (std::fread(p, 1, n, f) != n) return false;
    *crc = crc_update(*crc, p, n);
    return true;
}

}  // namespace

extern "C" uint32_t zero_crc32(const void* data, int64_t n) {
    std::call_once(g_crc_once, build_crc_table);
    if (!data || n <= 0) return 0u;
    return crc_update(0xFFFFFFFFu, data, (size_t)n) ^ 0xFFFFFFFFu;
}

extern "C" int zero_ckpt_write_shard(const char* path, const zero_ckpt_header_t* h,
                                     const float* master, const float* m, const float* v,
                                     const uint16_t* w_bf16) {
    std::call_once(g_crc_once, build_crc_table);
    if (!path || !h || !master || !m || !v) return ZERO_EINVAL;
    if (h->n_dp < 1 || h->rank < 0 || h->rank >= h->n_dp || h->shard < 0 || h->step < 0 ||
        h->shard > kMaxShardElems / h->n_dp ||                  // before the product can overflow
        h->padded_n != h->shard * (int64_t)h->n_dp || h->n < 0 || h->n > h->padded_n)
        return ZERO_EINVAL;
    FileHeader fh;
    std::memset(&fh, 0, sizeof fh);
    std::memcpy(fh.magic, kMagic, sizeof kMagic);
    fh.version = kVersion;
    fh.flags = w_bf16 ? 1u : 0u;
    fh.h = *h;
    const size_t s = (size_t)h->shard;
    // the payload CRC goes into the header: compute it first, then write
    uint32_t crc = 0xFFFFFFFFu;
    crc = crc_update(crc, master, s * 4);
    crc = crc_update(crc, m, s * 4);
    crc = crc_update(crc, v, s * 4);
    if (w_bf16) crc = crc_update(crc, w_bf16, s * 2);
    fh.crc = crc ^ 0xFFFFFFFFu;
    FILE* f = std::fopen(path, "wb");
    if (!f) return ZERO_EIO;
    bool ok = std::fwrite(&fh, 1, sizeof fh, f) == sizeof fh && write_all(f, master, s * 4) &&
              write_all(f, m, s * 4) && write_all(f, v, s * 4) && (!w_bf16 || write_all(f, w_bf16, s * 2));
    ok = (std::fclose(f) == 0) && ok;
    return ok ? ZERO_OK : ZERO_EIO;
}

extern "C" int zero_ckpt_read_header(const char* path, zero_ckpt_header_t* h, int32_t* has_bf16) {
    if (!path || !h) return ZERO_EINVAL;
    FILE* f = std::fopen(path, "rb");
    if (!f) return ZERO_EIO;
    FileHeader fh;
    const bool ok = std::fread(&fh, 1, sizeof fh, f) == sizeof fh;
    std::fclose(f);
    if (!ok || std::memcmp(fh.magic, kMagic, sizeof kMagic) != 0 || fh.version != kVersion)
        return ZERO_ECORRUPT;
    *h = fh.h;
    if (has_bf16) *has_bf16 = (fh.flags & 1u) ? 1 : 0;
    return ZERO_OK;
}

extern "C" int zero_ckpt_payload_crc(const char* path, uint32_t* crc) {
    if (!path || !crc) return ZERO_EINVAL;
    FILE* f = std::fopen(path, "rb");
    if (!f) return ZERO_EIO;
    FileHeader fh;
    const bool ok = std::fread(&fh, 1, sizeof fh, f) == sizeof fh;
    std::fclose(f);
    if (!ok || std::memcmp(fh.magic, kMagic, sizeof kMagic) != 0 || fh.version != kVersion)
        return ZERO_ECORRUPT;
    *crc = fh.crc;
    return ZERO_OK;
}

extern "C" int zero_ckpt_read_shard(const char* path, zero_ckpt_header_t* h, float* master,
                                    float* m, float* v, uint16_t* w_bf16, int64_t capacity) {
    std::call_once(g_crc_once, build_crc_table);
    if (!path || !h || !master || !m || !v) return ZERO_EINVAL;
    FILE* f = std::fopen(path, "rb");
    if (!f) return ZERO_EIO;
    FileHeader fh;
    int rc = ZERO_OK;
    if (std::fread(&fh, 1, sizeof fh, f) != sizeof fh ||
        std::memcmp(fh.magic, kMagic, sizeof kMagic) != 0 || fh.version != kVersion) {
        rc = ZERO_ECORRUPT;
    } else if (fh.h.shard < 0 || fh.h.shard > capacity || fh.h.shard > kMaxShardElems) {
        rc = ZERO_ERANGE;
    } else if (w_bf16 && !(fh.flags & 1u)) {
        rc = ZERO_EINVAL;   // asked for bf16 weights the file does not hold
    } else {
        const size_t s = (size_t)fh.h.shard;
        uint32_t crc = 0xFFFFFFFFu;
        bool ok = read_all(f, master, s * 4, &crc) && read_all(f, m, s * 4, &crc) &&
                  read_all(f, v, s * 4, &crc);
        if (ok && (fh.flags & 1u)) {
            if (w_bf16) {
                ok = read_all(f, w_bf16, s * 2, &crc);
            } else {   // still part of the CRC
                unsigned char buf[4096];
                size_t left = s * 2;
                while (ok && left) {
                    const size_t k = left < sizeof buf ? left : sizeof buf;
                    ok = read_all(f, buf, k, &crc);
                    left -= k;
                }
            }
        }
        if (!ok) rc = ZERO_ECORRUPT;
        else if ((crc ^ 0xFFFFFFFFu) != fh.crc) rc = ZERO_ECORRUPT;
        else *h = fh.h;
    }
    std::fclose(f);
    return rc;
}
