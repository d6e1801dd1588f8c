// hostmem_plan.h -- how repops_host_alloc sizes and aligns a request (plain
// C++, no CUDA: the allocator includes it, and a host test compiles it with g++).
#pragma once

#include <cstddef>
#include <cstdint>

namespace repops {

struct HostAllocPlan {
    size_t len;      // bytes mapped and registered (a multiple of `unit`)
    size_t align;    // alignment of the start
    size_t span;     // bytes reserved before trimming to an aligned start
    bool in_huge;    // advised MADV_HUGEPAGE and touched once per huge page
};

// `pg`: the base page size; `huge`: the transparent huge page size, equal to
// pg where huge pages are off.  A request of at least a quarter of a huge page
// is rounded up to whole huge pages at a huge-page-aligned start (reserving one
// huge page more, trimmed at both ends); a smaller one to whole base pages.
// False for a request no mapping can hold.
inline bool host_alloc_plan(uint64_t bytes, size_t pg, size_t huge, HostAllocPlan *p) {
    if (bytes == 0 || pg == 0 || huge < pg) return false;
    if (bytes > uint64_t(SIZE_MAX / 2) - huge) return false;
    p->in_huge = huge > pg && size_t(bytes) >= huge / 4;
    const size_t unit = p->in_huge ? huge : pg;
    p->len = (size_t(bytes) + unit - 1) / unit * unit;
    p->align = p->in_huge ? huge : pg;
    p->span = p->len + (p->in_huge ? huge : 0);
    return true;
}

// Where the aligned start falls in a reservation at `raw` (page aligned, of
// plan.span bytes), and what is unmapped before it and after its plan.len bytes.
inline void host_alloc_trim(uintptr_t raw, const HostAllocPlan &p, uintptr_t *start, size_t *head,
                            size_t *tail) {
    *start = (raw + p.align - 1) / p.align * p.align;
    *head = size_t(*start - raw);
    *tail = p.span - *head - p.len;
}

}  // namespace repops
