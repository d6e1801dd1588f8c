// hostmem.cu -- page-locked host memory in transparent huge pages for the
// host-buffer entry points (host code only).
//
// A copy engine reads pinned host memory through the host's address
// translation.  On a GB300's Grace host the base page is 64 KB, and copies out
// of buffers pinned in such pages ran anywhere from 8 to 212 GB/s once a
// step's buffers passed ~16 GiB, varying from pass to pass; buffers held in
// transparent huge pages (512 MB there) kept the link's 209-212 GB/s.  So this
// allocator maps anonymous memory at a huge-page-aligned address, advises it
// MADV_HUGEPAGE and registers it with CUDA (which faults every page in and
// locks it).
#include <sys/mman.h>
#include <unistd.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "hostmem_plan.h"
#include "internal.cuh"

namespace repops {
namespace {

struct HostBlocks {
    std::mutex mu;
    std::unordered_map<void *, size_t> len;   // start -> mapped length
};

HostBlocks &host_blocks() {
    static HostBlocks b;
    return b;
}

size_t page_size() {
    const long p = sysconf(_SC_PAGESIZE);
    return p > 0 ? size_t(p) : size_t(4096);
}

// Whether the kernel hands out transparent huge pages for madvised memory:
// its mode is "always" or "madvise", not "never" (unreadable: not assumed).
bool huge_pages_enabled() {
    char mode[128] = {0};
    FILE *f = std::fopen("/sys/kernel/mm/transparent_hugepage/enabled", "r");
    if (!f) return false;
    const size_t n = std::fread(mode, 1, sizeof(mode) - 1, f);
    std::fclose(f);
    mode[n] = 0;
    return std::strstr(mode, "[never]") == nullptr && std::strchr(mode, '[') != nullptr;
}

// The kernel's transparent huge page size (2 MiB when it does not say), or
// the base page size where huge pages are off: then nothing is rounded up.
size_t huge_page_size() {
    static size_t h = [] {
        const size_t pg = page_size();
        if (!huge_pages_enabled()) return pg;
        size_t v = 0;
        if (FILE *f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
            unsigned long long x = 0;
            if (std::fscanf(f, "%llu", &x) == 1) v = size_t(x);
            std::fclose(f);
        }
        if (v < pg || (v & (v - 1)) != 0) v = size_t(2) << 20;
        return v;
    }();
    return h;
}

}  // namespace
}  // namespace repops

using namespace repops;

extern "C" int repops_host_alloc(uint64_t bytes, void **ptr_out) {
    if (!ptr_out) return REPOPS_ERR_INVALID_ARG;
    *ptr_out = nullptr;
    if (bytes == 0) return REPOPS_OK;
    // At least a quarter of a huge page: whole huge pages (a 256 MiB buffer
    // mapped the ordinary way, below the 512 MB huge page of a 64 KB-page
    // host, was the one part of a step whose copies swung between 33.8 and
    // 114 ms); smaller: base pages (hostmem_plan.h).
    HostAllocPlan plan;
    if (!host_alloc_plan(bytes, page_size(), huge_page_size(), &plan)) return REPOPS_ERR_INVALID_ARG;
    const size_t len = plan.len, span = plan.span, huge = huge_page_size();
    const bool in_huge = plan.in_huge;
    void *raw = mmap(nullptr, span, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (raw == MAP_FAILED) return REPOPS_ERR_ALLOC;
    uintptr_t start = 0;
    size_t head = 0, tail = 0;
    host_alloc_trim(reinterpret_cast<uintptr_t>(raw), plan, &start, &head, &tail);
    if (head) munmap(raw, head);
    if (tail) munmap(reinterpret_cast<void *>(start + len), tail);
    void *p = reinterpret_cast<void *>(start);
#ifdef MADV_HUGEPAGE
    if (in_huge) {
        madvise(p, len, MADV_HUGEPAGE);   // advice only: ordinary pages if refused
        // one write per huge page faults each whole aligned range in at once
        // (the pages are zero either way)
        volatile unsigned char *q = static_cast<volatile unsigned char *>(p);
        for (size_t off = 0; off < len; off += huge) q[off] = 0;
    }
#endif
    const cudaError_t e = cudaHostRegister(p, len, cudaHostRegisterPortable);
    if (e != cudaSuccess) {
        munmap(p, len);
        return set_cuda_error(e);
    }
    {
        HostBlocks &b = host_blocks();
        std::lock_guard<std::mutex> g(b.mu);
        b.len[p] = len;
    }
    *ptr_out = p;
    return REPOPS_OK;
}

extern "C" int repops_host_free(void *ptr) {
    if (!ptr) return REPOPS_OK;
    size_t len = 0;
    {
        HostBlocks &b = host_blocks();
        std::lock_guard<std::mutex> g(b.mu);
        auto it = b.len.find(ptr);
        if (it == b.len.end()) return REPOPS_ERR_INVALID_ARG;
        len = it->second;
        b.len.erase(it);
    }
    const cudaError_t e = cudaHostUnregister(ptr);
    munmap(ptr, len);
    return e == cudaSuccess ? REPOPS_OK : set_cuda_error(e);
}
