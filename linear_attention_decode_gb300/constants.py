"""Enumeration values of include/gdnreplay.h, shared by the binding and the input generators."""
import torch

# gdn_dtype_t
F32, BF16, F16 = 0, 1, 2
# gdn_gate_t
GATE_SCALAR, GATE_PER_K = 0, 1
# gdn_recon_t
RECON_TENSOR, RECON_FFMA, RECON_OUTPUT = 0, 1, 2
# gdn_step_t.flags bits
STEP_OVERLAP_PREVIOUS, STEP_PERSISTENT_KERNEL = 1, 2
# dev_status bits
DEV_BAD_SLOT, DEV_BAD_WRITE_POS, DEV_TIMEOUT, DEV_INTERNAL, DEV_BAD_ACCEPTED = 1, 2, 4, 8, 16

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}
GDN_DTYPE = {v: k for k, v in TORCH_DTYPE.items()}
