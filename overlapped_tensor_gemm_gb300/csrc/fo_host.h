// Host services of fo_api.cu used by the other host modules (not public ABI).
#pragma once

#include "fo_internal.h"

namespace fo {
fo_status host_buffer(fo_ctx* ctx, int slot, size_t bytes, void** out);  // attention workspace slots 0..7
fo_status host_flags(fo_ctx* ctx, uint32_t** out);                       // arrival flags [rank*P + slice]
uint32_t host_next_epoch(fo_ctx* ctx);
uint32_t* host_ctrl(fo_ctx* ctx);
int host_num_sms(fo_ctx* ctx);
cudaStream_t host_link(fo_ctx* ctx, int r);
cudaEvent_t host_ev_hop(fo_ctx* ctx, int r, int t);
fo_status host_fork(fo_ctx* ctx, int P, cudaStream_t s);
fo_status host_join(fo_ctx* ctx, int P, cudaStream_t s);
fo_status host_copy_rows(void* dst, int64_t dld, const void* src, int64_t sld, int64_t rows, int64_t cols,
                         size_t esz, cudaStream_t s);
fo_status host_write_flag(cudaStream_t s, uint32_t* flag, uint32_t value);
fo_status host_encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                          CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
fo_status host_check_mat(const fo_mat& a, int32_t dtype, const char* what, int r);
fo_status host_fail(fo_status st, const char* msg);
bool host_copies_first();  // host order of a ring's copies and the kernel that waits on them
uint64_t host_timeout_ns(const fo_opts& o);
int host_grid(fo_ctx* ctx, const fo_opts& o, int work);
void host_phase_record(fo_ctx* ctx, int i, cudaStream_t s);     // serial baselines' phase events
void host_phase_done(fo_ctx* ctx, bool gemm_first);
}  // namespace fo
