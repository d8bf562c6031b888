"""Host-side structure of the fused launch, checked without a GPU.

The fused kernel needs more than 48 KB of dynamic shared memory, which CUDA
grants per device and per kernel (cudaFuncSetAttribute). A process-wide
"already set" flag would leave a second device without it, and its fused
launches would fail; the launch therefore sets the attribute on every call,
for the device current at that call. Only one device is available to the GPU
tests, so this file checks the launch code itself: the attribute call sits in
fused_launch, on the path to the kernel launch, with no once-only guard."""

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tp_vocab_logits_gb300", "csrc", "hg_fused.cu")


def function_body(src: str, signature: str) -> str:
    start = src.index(signature)
    i = src.index("{", start)
    depth = 0
    for j in range(i, len(src)):
        if src[j] == "{":
            depth += 1
        elif src[j] == "}":
            depth -= 1
            if depth == 0:
                return src[i:j + 1]
    raise AssertionError(f"unbalanced braces after {signature}")


def code_only(text: str) -> str:
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def test_fused_launch_sets_the_shared_memory_attribute_on_every_call():
    src = code_only(open(SRC).read())
    body = function_body(src, "cudaError_t fused_launch(")
    set_at = body.find("cudaFuncSetAttribute(fused_kernel")
    launch_at = body.find("cudaLaunchKernelEx")
    assert set_at >= 0, "fused_launch no longer sets the dynamic shared-memory attribute"
    assert launch_at > set_at, "the attribute must be set before the launch"
    assert "cudaFuncAttributeMaxDynamicSharedMemorySize" in body[set_at:launch_at]
    # Nothing may skip it on a later call: no static state in the function and
    # no branch between the function's start and the attribute call.
    assert not re.search(r"\bstatic\b", body), "static state in fused_launch"
    assert not re.search(r"\b(if|for|while|switch)\b", body[:set_at]), \
        "the attribute call is conditional"


def test_no_once_only_flag_for_the_attribute_anywhere():
    src = code_only(open(SRC).read())
    calls = [m.start() for m in re.finditer(r"cudaFuncSetAttribute\(", src)]
    assert len(calls) == 1, "expected exactly one attribute call (in fused_launch)"
    assert not re.search(r"\bstatic\s+(bool|int|std::atomic<bool>|std::once_flag)\b", src), \
        "a file-scope once-only flag"
