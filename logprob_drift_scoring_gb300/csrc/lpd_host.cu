// Page-locked host memory for the host-input scoring path (lpd_score_host).
//
// The host-to-device link is the bound of scoring logits that live in host
// memory, so the staging memory should let the copy engines run at the link
// rate with as few page translations as possible: an anonymous mapping
// advised for transparent huge pages, then registered with the runtime.
// Registration faults the pages in, so the advice takes effect before any
// copy.
#include <sys/mman.h>

#include "lpd_internal.cuh"

extern "C" {

void *lpd_host_alloc(size_t bytes) {
    if (bytes == 0) return nullptr;
    void *p = mmap(nullptr, bytes, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p == MAP_FAILED) return nullptr;
#ifdef MADV_HUGEPAGE
    madvise(p, bytes, MADV_HUGEPAGE);  // advice only: without it the pages are just smaller
#endif
    if (cudaHostRegister(p, bytes, cudaHostRegisterDefault) != cudaSuccess) {
        cudaGetLastError();  // leave no sticky error behind for the caller's next call
        munmap(p, bytes);
        return nullptr;
    }
    return p;
}

int lpd_host_free(void *ptr, size_t bytes) {
    if (!ptr) return LPD_ERR_NULL_POINTER;
    const cudaError_t e = cudaHostUnregister(ptr);
    munmap(ptr, bytes);
    return e == cudaSuccess ? LPD_OK : LPD_ERR_CUDA;
}

}  // extern "C"
