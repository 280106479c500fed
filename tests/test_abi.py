"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/pkv.h declares.  Host-side argument checks are exercised only where
they return before any CUDA call (no GPU here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_29_gb300 import build
    build.build()
    import paged_kv_attention_29_gb300 as pkv
    return pkv.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PKV_API\s+[\w\s\*]*?\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_symbols()
    for must in ["pkv_slot_mapping", "pkv_store_kvcache", "pkv_prefill_varlen", "pkv_prefill_plan",
                 "pkv_prefill_varlen_planned", "pkv_decode", "pkv_sample",
                 "pkv_decode_workspace_size", "pkv_get_device_error", "pkv_status_string"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_build_targets_sm103a_only():
    from paged_kv_attention_29_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    import paged_kv_attention_29_gb300 as pkv
    assert pkv.pkv_status_string(0) == "PKV_OK"
    assert pkv.pkv_status_string(3) == "PKV_ERR_WORKSPACE"
    assert pkv.pkv_abi_version() == 1


def test_host_argument_checks_return_before_launch(lib):
    P = None
    # store: negative token count; row stride smaller than a row
    assert lib.pkv_store_kvcache(P, P, -1, 1024, 1024, P, P, P, 4, 256, 8, 128, P) == 1
    assert lib.pkv_store_kvcache(P, P, 4, 512, 1024, P, P, P, 4, 256, 8, 128, P) == 1
    # decode: unsupported head_dim / group (3 and 16 query heads per KV head) / block size
    assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, 16, 8, 64, 256, 4, 0.1, P, P, 0, P) == 2
    assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, 12, 4, 128, 256, 4, 0.1, P, P, 0, P) == 2
    assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, 16, 1, 128, 256, 4, 0.1, P, P, 0, P) == 2
    assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, 16, 8, 128, 100, 4, 0.1, P, P, 0, P) == 2
    # every supported group (1, 2, 4, 8) passes the shape check and stops at the null pointers
    for hq, hkv in ((16, 16), (16, 8), (16, 4), (16, 2), (32, 4), (8, 1)):
        assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, hq, hkv, 128, 256, 4, 0.1, P, P, 0, P) == 1
        assert lib.pkv_prefill_varlen(P, P, P, P, P, P, 4, 2, 10, 9, 9, hq, hkv, 128, 256, 4, 0.1, P, P, 0, P) == 1
        assert lib.pkv_prefill_workspace_size(4, hq, hkv, 128, 100) > 0
    assert lib.pkv_prefill_varlen(P, P, P, P, P, P, 4, 2, 10, 9, 9, 12, 4, 128, 256, 4, 0.1, P, P, 0, P) == 2
    assert lib.pkv_prefill_workspace_size(4, 12, 4, 128, 100) == 0
    assert lib.pkv_decode_workspace_size(4, 12, 4, 128) == 0
    # decode, decode_append: a softmax scale that is not a positive finite number
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        assert lib.pkv_decode(P, P, P, P, 4, P, 2, 10, 16, 8, 128, 256, 4, bad, P, P, 0, P) == 1
        assert lib.pkv_decode_append(P, P, P, P, P, P, 4, P, 2, 10, 16, 8, 128, 256, 4, bad, P, P, P, 0, P) == 1
    # prefill: max_seqlen_q > max_seqlen_k
    assert lib.pkv_prefill_varlen(P, P, P, P, P, P, 4, 2, 10, 9, 8, 16, 8, 128, 256, 4, 0.1, P, P, 0, P) == 1
    # planned prefill: the plan checks the arguments it takes, the planned call those of pkv_prefill_varlen
    assert lib.pkv_prefill_plan(P, P, 4, 2, 10, 9, 9, 16, 8, 128, 256, P, 0, P) == 1        # null cu_seqlens
    assert lib.pkv_prefill_plan(P, P, 4, 2, 10, 9, 9, 12, 4, 128, 256, P, 0, P) == 2        # group of 3
    assert lib.pkv_prefill_plan(P, P, 4, 2, 10, 9, 8, 16, 8, 128, 256, P, 0, P) == 1        # max_q > max_k
    assert lib.pkv_prefill_plan(P, P, 4, 0, 10, 9, 9, 16, 8, 128, 256, P, 0, P) == 0        # no sequences
    assert lib.pkv_prefill_varlen_planned(P, P, P, P, P, P, 4, 2, 10, 9, 9, 16, 8, 128, 256, 4, 0.1, P, P, 0, P) == 1
    assert lib.pkv_prefill_varlen_planned(P, P, P, P, P, P, 4, 2, 10, 9, 9, 16, 8, 128, 256, 4, 0.0, P, P, 0, P) == 1
    assert lib.pkv_prefill_varlen_planned(P, P, P, P, P, P, 4, 2, 10, 9, 9, 12, 4, 128, 256, 4, 0.1, P, P, 0, P) == 2
    # slot mapping: both or neither of cu_seqlens_k / context_lens
    assert lib.pkv_slot_mapping(P, P, P, P, 4, 2, 2, 256, 4, P, P) == 1
    # sample: row stride below vocab, empty vocab
    assert lib.pkv_sample(P, 2, 100, 50, P, 0, 0, P, P) == 1
    assert lib.pkv_sample(P, 2, 0, 0, P, 0, 0, P, P) == 1
    # rope+store: head_dim not a multiple of 16; q without q_out; base <= 0; strides below a row
    assert lib.pkv_rope_store_kvcache(P, 0, P, 0, P, 800, P, 800, P, 4, 0, 8, 100, 1e6, P, P, P, 4, 256, P) == 2
    fake_q = ctypes.c_void_p(16)    # non-null, never dereferenced: the check returns first
    assert lib.pkv_rope_store_kvcache(fake_q, 2048, P, 2048, P, 1024, P, 1024, P, 4, 16, 8, 128, 1e6,
                                      P, P, P, 4, 256, P) == 1
    assert lib.pkv_rope_store_kvcache(P, 0, P, 0, P, 1024, P, 1024, P, 4, 0, 8, 128, 0.0, P, P, P, 4, 256, P) == 1
    assert lib.pkv_rope_store_kvcache(P, 0, P, 0, P, 512, P, 1024, P, 4, 0, 8, 128, 1e6, P, P, P, 4, 256, P) == 1
    assert lib.pkv_rope_store_kvcache(P, 0, P, 0, P, 1024, P, 1024, P, 0, 0, 8, 128, 1e6, P, P, P, 4, 256, P) == 0
    # decode_append: unsupported head_dim; a pointer that is not 16-byte aligned; zero batch is a no-op
    assert lib.pkv_decode_append(P, P, P, P, P, P, 4, P, 2, 10, 16, 8, 64, 256, 4, 0.1, P, P, P, 0, P) == 2
    odd = ctypes.c_void_p(8)        # non-null, 8-byte aligned only, never dereferenced
    assert lib.pkv_decode_append(odd, odd, odd, odd, odd, odd, 4, odd, 2, 10, 16, 8, 128, 256, 4, 0.1, odd, P, P, 0,
                                 P) == 2
    assert lib.pkv_decode_append(P, P, P, P, P, P, 4, P, 0, 10, 16, 8, 128, 256, 4, 0.1, P, P, P, 0, P) == 0
    # zero-size calls are no-ops
    assert lib.pkv_store_kvcache(P, P, 0, 1024, 1024, P, P, P, 4, 256, 8, 128, P) == 0
    assert lib.pkv_sample(P, 0, 10, 10, P, 0, 0, P, P) == 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import paged_kv_attention_29_gb300 as pkv
    x = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    pool = torch.zeros(2, 256, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.pkv_store_kvcache(x, x, torch.zeros(4, dtype=torch.int32), pool, pool)


def test_readme_example_calls_the_binding_as_it_is():
    """Every pkv.* call in the README's Python example names a binding function and passes
    arguments its signature accepts."""
    import ast
    import inspect
    import paged_kv_attention_29_gb300 as pkv
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "the README has no Python example"
    calls = [n for b in blocks for n in ast.walk(ast.parse(b))
             if isinstance(n, ast.Call) and isinstance(n.func, ast.Attribute)
             and isinstance(n.func.value, ast.Name) and n.func.value.id == "pkv"]
    assert len(calls) >= 5
    for c in calls:
        fn = getattr(pkv, c.func.attr)
        sig = inspect.signature(fn)
        args = [object()] * len(c.args)
        kwargs = {k.arg: object() for k in c.keywords}
        sig.bind(*args, **kwargs)        # raises TypeError on a wrong name or count
