"""Rules the CUDA sources keep, checked by a scan (no GPU): no kernel can trap
or fail a device assertion (device failures are reported through the status
word instead), and every loop that spins on an mbarrier has a time limit."""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "w8a8_quantized_projections_gb300", "csrc")


def _code(path):
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)      # block comments
    return re.sub(r"//[^\n]*", "", text)                     # line comments


def _files():
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".cu", ".cuh", ".h"))]


def test_no_trap_or_device_assert():
    for path in _files():
        code = _code(path)
        assert "trap" not in code, path
        assert not re.search(r"(?<!static_)\bassert\s*\(", code), path


def _innermost_loop(code, pos):
    """Text of the innermost for/while loop body enclosing pos, or None."""
    stack, blocks = [], []
    for i, ch in enumerate(code[:pos]):
        if ch == "{":
            stack.append(i)
        elif ch == "}" and stack:
            stack.pop()
    for start in reversed(stack):
        # the block's header: `keyword (...)` right before the brace
        j = start - 1
        while j >= 0 and code[j].isspace():
            j -= 1
        if j < 0 or code[j] != ")":
            continue
        depth = 0
        while j >= 0:
            depth += (code[j] == ")") - (code[j] == "(")
            if depth == 0:
                break
            j -= 1
        m = re.search(r"\b(\w+)\s*$", code[max(0, j - 40):j])
        if m and m.group(1) in ("for", "while"):
            depth, j = 0, start
            while j < len(code):
                depth += (code[j] == "{") - (code[j] == "}")
                if depth == 0:
                    return code[start:j]
                j += 1
    return None


def test_every_mbarrier_spin_is_time_limited():
    """Each loop that polls an mbarrier (a *try_wait* call inside a for/while
    body) also reads the global timer to give up after a limit."""
    calls = 0
    for path in _files():
        code = re.sub(r'"[^"\n]*"', '""', _code(path))       # drop asm strings
        for m in re.finditer(r"\b\w*try_wait\w*\s*\(", code):
            line_start = code.rfind("\n", 0, m.start()) + 1
            if re.match(r"\s*(__device__|static|template|inline)", code[line_start:m.start()]):
                continue                                      # the helper's definition
            body = _innermost_loop(code, m.start())
            if body is None:
                continue                                      # a single poll, no spin
            calls += 1
            assert "globaltimer_ns()" in body, (path, code[line_start:m.end() + 40])
    assert calls >= 4


def test_every_endless_loop_form_has_a_time_limit():
    """Loops written without an exit condition (`for (..;;..)`, `while (1)`,
    `while (true)`) must read the global timer in their body."""
    n = 0
    for path in _files():
        code = _code(path)
        for m in re.finditer(r"\bfor\s*\([^;()]*;\s*;[^)]*\)\s*\{|\bwhile\s*\(\s*(1|true)\s*\)\s*\{", code):
            body = _innermost_loop(code, m.end())
            assert body is not None and "globaltimer_ns()" in body, (path, m.group(0))
            n += 1
    assert n >= 4
