"""The Python binding's buffer-size checks, on the CPU.  The C entry points
take bare pointers and cannot see how large a buffer is, so the binding
refuses any output, index or input buffer too small for the call before it
takes a pointer.  With CPU tensors a call whose sizes are right gets as far as
taking pointers and stops there ("expected a CUDA tensor"), which shows the
checks let it through."""
import pytest
import torch

import moe_token_permute_gb300 as mp
from moe_token_permute_gb300 import build as cuda_build

T, K, E, EL, H, S, M = 6, 2, 8, 4, 256, 2, 5
R = T * K


@pytest.fixture(scope="module", autouse=True)
def built():
    cuda_build.build()


def i32(*shape):
    return torch.zeros(*shape, dtype=torch.int32)


def permute_args(**over):
    a = dict(hidden_states=torch.zeros(T, H, dtype=torch.bfloat16), topk_ids=i32(T, K),
             expert_first_token_offset=torch.zeros(EL + 1, dtype=torch.int64),
             permuted_idx=i32(R), inv_permuted_idx=i32(R),
             workspace=torch.zeros(1 << 16, dtype=torch.uint8), num_experts=E,
             num_local_experts=EL, expert_map=i32(E),
             hidden_scales=torch.zeros(T, S), permuted_hidden_states=torch.zeros(R, H, dtype=torch.bfloat16),
             permuted_scales=torch.zeros(R, S))
    a.update(over)
    return a


def call_permute(**over):
    a = permute_args(**over)
    return mp.moe_permute(a.pop("hidden_states"), a.pop("topk_ids"),
                          a.pop("expert_first_token_offset"), a.pop("permuted_idx"),
                          a.pop("inv_permuted_idx"), a.pop("workspace"), **a)


def test_permute_right_sizes_reach_the_pointers():
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_permute()
    # larger buffers than needed are fine too
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_permute(permuted_idx=i32(R + 3), hidden_states=torch.zeros(T + 2, H, dtype=torch.bfloat16))


@pytest.mark.parametrize("over,what", [
    (dict(permuted_idx=i32(R - 1)), "permuted_idx"),
    (dict(inv_permuted_idx=i32(R - 1)), "inv_permuted_idx"),
    (dict(expert_first_token_offset=torch.zeros(EL, dtype=torch.int64)), "expert_first_token_offset"),
    (dict(expert_map=i32(E - 1)), "expert_map"),
    (dict(hidden_states=torch.zeros(T - 1, H, dtype=torch.bfloat16)), "hidden_states"),
    (dict(hidden_states=torch.zeros(T * H, dtype=torch.bfloat16)), "hidden_states"),
    (dict(permuted_hidden_states=torch.zeros(R - 1, H, dtype=torch.bfloat16)), "permuted_hidden_states"),
    # same element count but half the bytes of the source rows
    (dict(permuted_hidden_states=torch.zeros(R, H, dtype=torch.uint8)), "permuted_hidden_states"),
    (dict(hidden_scales=torch.zeros(T - 1, S)), "hidden_scales"),
    (dict(permuted_scales=torch.zeros(R - 1, S)), "permuted_scales"),
])
def test_permute_refuses_small_buffers(over, what):
    with pytest.raises(ValueError, match=what):
        call_permute(**over)


def call_batched(**over):
    a = dict(hidden_states=torch.zeros(T, H, dtype=torch.bfloat16), topk_ids=i32(T, K),
             expert_num_tokens=i32(EL), inv_permuted_idx=i32(R),
             workspace=torch.zeros(1 << 16, dtype=torch.uint8), num_experts=E,
             max_rows_per_expert=M, num_local_experts=EL, expert_map=i32(E),
             hidden_scales=torch.zeros(T, S),
             batched_hidden_states=torch.zeros(EL, M, H, dtype=torch.bfloat16),
             batched_scales=torch.zeros(EL * M, S))
    a.update(over)
    return mp.moe_permute_batched(a.pop("hidden_states"), a.pop("topk_ids"),
                                  a.pop("expert_num_tokens"), a.pop("inv_permuted_idx"),
                                  a.pop("workspace"), **a)


def test_batched_right_sizes_reach_the_pointers():
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_batched()


@pytest.mark.parametrize("over,what", [
    (dict(expert_num_tokens=i32(EL - 1)), "expert_num_tokens"),
    (dict(inv_permuted_idx=i32(R - 1)), "inv_permuted_idx"),
    (dict(expert_map=i32(E - 1)), "expert_map"),
    (dict(hidden_states=torch.zeros(T - 1, H, dtype=torch.bfloat16)), "hidden_states"),
    (dict(batched_hidden_states=torch.zeros(EL, M - 1, H, dtype=torch.bfloat16)), "batched_hidden_states"),
    (dict(batched_scales=torch.zeros(EL * M - 1, S)), "batched_scales"),
])
def test_batched_refuses_small_buffers(over, what):
    with pytest.raises(ValueError, match=what):
        call_batched(**over)


def call_quant(**over):
    a = dict(hidden_states=torch.zeros(T, H, dtype=torch.bfloat16), topk_ids=i32(T, K),
             expert_first_token_offset=torch.zeros(EL + 1, dtype=torch.int64),
             permuted_idx=i32(R), inv_permuted_idx=i32(R),
             workspace=torch.zeros(1 << 16, dtype=torch.uint8),
             permuted_codes=torch.zeros(R, H, dtype=torch.uint8),
             permuted_scales=torch.zeros(R, H // 128), num_experts=E, num_local_experts=EL,
             expert_map=i32(E))
    a.update(over)
    return mp.moe_permute_quant_fp8(a.pop("hidden_states"), a.pop("topk_ids"),
                                    a.pop("expert_first_token_offset"), a.pop("permuted_idx"),
                                    a.pop("inv_permuted_idx"), a.pop("workspace"),
                                    a.pop("permuted_codes"), a.pop("permuted_scales"), **a)


def test_quant_right_sizes_reach_the_pointers():
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_quant()


@pytest.mark.parametrize("over,what", [
    (dict(permuted_codes=torch.zeros(R - 1, H, dtype=torch.uint8)), "permuted_codes"),
    (dict(permuted_scales=torch.zeros(R, H // 128 - 1)), "permuted_scales"),
    (dict(permuted_idx=i32(R - 1)), "permuted_idx"),
    (dict(inv_permuted_idx=i32(2)), "inv_permuted_idx"),
    (dict(expert_first_token_offset=torch.zeros(2, dtype=torch.int64)), "expert_first_token_offset"),
    (dict(expert_map=i32(3)), "expert_map"),
    (dict(hidden_states=torch.zeros(T - 2, H, dtype=torch.bfloat16)), "hidden_states"),
])
def test_quant_refuses_small_buffers(over, what):
    with pytest.raises(ValueError, match=what):
        call_quant(**over)


def call_unpermute(**over):
    a = dict(permuted_rows=torch.zeros(R, H, dtype=torch.bfloat16), topk_weights=torch.zeros(T, K),
             inv_permuted_idx=i32(R), out=torch.zeros(T, H, dtype=torch.bfloat16))
    a.update(over)
    return mp.moe_unpermute(a["permuted_rows"], a["topk_weights"], a["inv_permuted_idx"], a["out"])


def test_unpermute_right_sizes_reach_the_pointers():
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_unpermute()
    # fewer expert rows than T*K is legal (dropped rows are never read)
    with pytest.raises(ValueError, match="CUDA tensor"):
        call_unpermute(permuted_rows=torch.zeros(3, H, dtype=torch.bfloat16))


@pytest.mark.parametrize("over,what", [
    (dict(out=torch.zeros(T - 1, H, dtype=torch.bfloat16)), "out"),
    (dict(inv_permuted_idx=i32(R - 1)), "inv_permuted_idx"),
])
def test_unpermute_refuses_small_buffers(over, what):
    with pytest.raises(ValueError, match=what):
        call_unpermute(**over)


@pytest.mark.parametrize("dst,msg", [
    (torch.zeros(1, dtype=torch.float32), "32-bit integer"),   # not an integer
    (torch.zeros(1, dtype=torch.int64), "32-bit integer"),     # 8-byte elements
    (torch.zeros(0, dtype=torch.int32), "32-bit integer"),     # no room for the word
    (torch.zeros(4, dtype=torch.int32)[::2], "contiguous"),
    (torch.zeros(1, dtype=torch.int32), "pinned host memory"),  # pageable host memory
])
def test_async_status_read_refuses_unusable_destinations(dst, msg):
    """moe_permute_read_status writes the status word through dst from a
    kernel: dst must be one 32-bit word of device or pinned host memory, which
    the binding checks before taking any pointer."""
    ws = torch.zeros(1 << 12, dtype=torch.uint8)
    with pytest.raises(ValueError, match=msg):
        mp.moe_permute_read_status(ws, dst)
