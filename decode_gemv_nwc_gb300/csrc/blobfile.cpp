// blobfile.cpp -- compressed checkpoints: named NWC blobs in one file, and loading one of them
// straight into caller-owned device memory (the NWC page's usage block: a compressed model is
// saved once and later loaded onto the GPU without the BF16 originals).
//
// File layout (little-endian): "NWCF", u32 entry count, then per entry a u32 name length, the
// UTF-8 name (1..4096 bytes, unique within the file), a u64 blob length, zero bytes up to the
// next 16-byte file offset, and the blob. The file ends with the last blob. Blob starts are
// 16-byte aligned in the file so that a reader may map or stream it straight into aligned
// buffers.
//
// Every entry is validated (nwc_validate) on the way in and on the way out; the index walk
// checks every length against the file size before reading, so a truncated or garbled file
// is NWC_ERR_FORMAT, never an out-of-bounds read.
#include <cuda_runtime_api.h>

#include <cstdio>
#include <cstring>
#include <string>
#include <unordered_set>
#include <vector>

#include "nwc.h"

namespace {

constexpr char kFileMagic[4] = {'N', 'W', 'C', 'F'};
constexpr uint32_t kMaxName = 4096;
constexpr uint32_t kMaxEntries = 1u << 20;

uint64_t up16(uint64_t a) { return (a + 15) & ~uint64_t(15); }

struct File {
    std::FILE *f = nullptr;
    ~File() {
        if (f) std::fclose(f);
    }
};

struct Entry {
    std::string name;
    uint64_t offset, bytes;
};

bool read_at(std::FILE *f, uint64_t pos, void *dst, size_t n) {
    if (fseeko(f, (off_t)pos, SEEK_SET) != 0) return false;
    return std::fread(dst, 1, n, f) == n;
}

// Index of the file at path: every entry's name, blob offset and length. NWC_ERR_IO for a
// file that cannot be opened, NWC_ERR_FORMAT for one whose structure does not hold.
nwc_status read_index(const char *path, std::vector<Entry> &out) {
    if (!path) return NWC_ERR_INVALID_ARG;
    File h;
    h.f = std::fopen(path, "rb");
    if (!h.f) return NWC_ERR_IO;
    if (fseeko(h.f, 0, SEEK_END) != 0) return NWC_ERR_FORMAT;
    const off_t end = ftello(h.f);
    if (end < 8) return NWC_ERR_FORMAT;
    const uint64_t size = (uint64_t)end;
    uint8_t head[8];
    if (!read_at(h.f, 0, head, 8) || std::memcmp(head, kFileMagic, 4) != 0) return NWC_ERR_FORMAT;
    uint32_t count;
    std::memcpy(&count, head + 4, 4);
    if (count > kMaxEntries) return NWC_ERR_FORMAT;
    out.clear();
    out.reserve(count);
    std::unordered_set<std::string> seen;
    uint64_t pos = 8;
    for (uint32_t i = 0; i < count; i++) {
        uint32_t len;
        if (pos + 4 > size || !read_at(h.f, pos, &len, 4)) return NWC_ERR_FORMAT;
        if (len == 0 || len > kMaxName || pos + 4 + len + 8 > size) return NWC_ERR_FORMAT;
        Entry e;
        e.name.resize(len);
        uint64_t blen;
        if (!read_at(h.f, pos + 4, &e.name[0], len) || !read_at(h.f, pos + 4 + len, &blen, 8)) return NWC_ERR_FORMAT;
        if (std::memchr(e.name.data(), 0, len)) return NWC_ERR_FORMAT;
        const uint64_t start = up16(pos + 4 + len + 8);
        if (start > size || blen > size - start) return NWC_ERR_FORMAT;
        if (!seen.insert(e.name).second) return NWC_ERR_FORMAT;
        e.offset = start;
        e.bytes = blen;
        out.push_back(std::move(e));
        pos = start + blen;
    }
    return pos == size ? NWC_OK : NWC_ERR_FORMAT;
}

// Reads entry `index` into blob_host (capacity cap) and validates it.
nwc_status read_entry(const char *path, int index, void *blob_host, size_t cap, size_t *bytes, std::vector<Entry> &idx) {
    nwc_status st = read_index(path, idx);
    if (st != NWC_OK) return st;
    if (index < 0 || (size_t)index >= idx.size()) return NWC_ERR_INVALID_ARG;
    const Entry &e = idx[(size_t)index];
    if (bytes) *bytes = e.bytes;
    if (!blob_host || cap < e.bytes) return NWC_ERR_INVALID_ARG;
    File h;
    h.f = std::fopen(path, "rb");
    if (!h.f) return NWC_ERR_IO;
    if (!read_at(h.f, e.offset, blob_host, e.bytes)) return NWC_ERR_IO;
    return nwc_validate(blob_host, e.bytes);
}

}  // namespace

extern "C" nwc_status nwc_file_save(const char *path, int count, const char *const *names,
                                    const void *const *blobs, const size_t *bytes) {
    if (!path || count < 0 || (uint32_t)count > kMaxEntries) return NWC_ERR_INVALID_ARG;
    if (count > 0 && (!names || !blobs || !bytes)) return NWC_ERR_INVALID_ARG;
    std::unordered_set<std::string> seen;
    for (int i = 0; i < count; i++) {
        if (!names[i] || !blobs[i]) return NWC_ERR_INVALID_ARG;
        const size_t len = std::strlen(names[i]);
        if (len == 0 || len > kMaxName || !seen.insert(names[i]).second) return NWC_ERR_INVALID_ARG;
        nwc_status st = nwc_validate(blobs[i], bytes[i]);
        if (st != NWC_OK) return st;
    }
    // written next to the target, then renamed over it: a reader never sees a partial file
    const std::string tmp = std::string(path) + ".partial";
    File h;
    h.f = std::fopen(tmp.c_str(), "wb");
    if (!h.f) return NWC_ERR_IO;
    static const uint8_t zeros[16] = {0};
    bool ok = std::fwrite(kFileMagic, 1, 4, h.f) == 4;
    const uint32_t c = (uint32_t)count;
    ok = ok && std::fwrite(&c, 4, 1, h.f) == 1;
    uint64_t pos = 8;
    for (int i = 0; ok && i < count; i++) {
        const uint32_t len = (uint32_t)std::strlen(names[i]);
        const uint64_t blen = bytes[i];
        ok = std::fwrite(&len, 4, 1, h.f) == 1 && std::fwrite(names[i], 1, len, h.f) == len &&
             std::fwrite(&blen, 8, 1, h.f) == 1;
        pos += 4 + len + 8;
        const size_t pad = (size_t)(up16(pos) - pos);
        ok = ok && std::fwrite(zeros, 1, pad, h.f) == pad && std::fwrite(blobs[i], 1, blen, h.f) == blen;
        pos += pad + blen;
    }
    ok = ok && std::fflush(h.f) == 0;
    ok = (std::fclose(h.f) == 0) && ok;
    h.f = nullptr;
    if (!ok || std::rename(tmp.c_str(), path) != 0) {
        std::remove(tmp.c_str());
        return NWC_ERR_IO;
    }
    return NWC_OK;
}

extern "C" nwc_status nwc_file_count(const char *path, int *count) {
    if (!count) return NWC_ERR_INVALID_ARG;
    std::vector<Entry> idx;
    nwc_status st = read_index(path, idx);
    if (st == NWC_OK) *count = (int)idx.size();
    return st;
}

extern "C" nwc_status nwc_file_entry(const char *path, int index, char *name, size_t name_cap, size_t *bytes) {
    std::vector<Entry> idx;
    nwc_status st = read_index(path, idx);
    if (st != NWC_OK) return st;
    if (index < 0 || (size_t)index >= idx.size()) return NWC_ERR_INVALID_ARG;
    const Entry &e = idx[(size_t)index];
    if (bytes) *bytes = e.bytes;
    if (name) {
        if (name_cap < e.name.size() + 1) return NWC_ERR_INVALID_ARG;
        std::memcpy(name, e.name.c_str(), e.name.size() + 1);
    }
    return NWC_OK;
}

extern "C" nwc_status nwc_file_find(const char *path, const char *name, int *index) {
    if (!name || !index) return NWC_ERR_INVALID_ARG;
    std::vector<Entry> idx;
    nwc_status st = read_index(path, idx);
    if (st != NWC_OK) return st;
    for (size_t i = 0; i < idx.size(); i++)
        if (idx[i].name == name) {
            *index = (int)i;
            return NWC_OK;
        }
    return NWC_ERR_INVALID_ARG;
}

extern "C" nwc_status nwc_file_read(const char *path, int index, void *blob_host, size_t cap, size_t *bytes) {
    std::vector<Entry> idx;
    return read_entry(path, index, blob_host, cap, bytes, idx);
}

extern "C" nwc_status nwc_file_load(const char *path, int index, void *blob_host, size_t host_cap, void *blob_dev,
                                    size_t dev_cap, nwc_matrix *out, nwc_stream stream) {
    if (!blob_dev || !out) return NWC_ERR_INVALID_ARG;
    std::vector<Entry> idx;
    size_t bytes = 0;
    nwc_status st = read_entry(path, index, blob_host, host_cap, &bytes, idx);
    if (st != NWC_OK) return st;
    if (dev_cap < bytes) return NWC_ERR_INVALID_ARG;
    nwc_matrix m;
    st = nwc_bind(blob_host, bytes, blob_dev, &m);
    if (st != NWC_OK) return st;
    if (cudaMemcpyAsync(blob_dev, blob_host, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream) != cudaSuccess)
        return NWC_ERR_CUDA;
    *out = m;
    return NWC_OK;
}
