"""Host logic of bench.py that needs no GPU: the check that keeps a recorded DRAM figure tied to
the kernel code it was taken on."""
import bench


def test_code_hash_ignores_comments_only(tmp_path):
    """The recorded DRAM traffic stays valid across comment edits of the kernel source, and only
    those: a change in code or in a string literal (inline PTX) gives another hash."""
    src = open(bench.KERNEL_SRC, encoding="utf-8").read()
    base = bench.code_sha256(bench.KERNEL_SRC)

    def h(text):
        p = tmp_path / "k.cu"
        p.write_text(text, encoding="utf-8")
        return bench.code_sha256(str(p))

    assert h(src) == base
    assert h(src.replace("// ---", "// ---- edited ", 1)) == base
    assert h("/* a block comment */\n" + src + "\n// trailing\n") == base
    assert h(src.replace("red.shared.add.u32", "red.shared.add.s32", 1)) != base
    assert h(src.replace("kThreads", "kThreads + 0", 1)) != base


def test_code_hash_covers_the_schedule_header(tmp_path):
    """The recorded figure is tied to the draw placement too (csrc/schedule.h)."""
    base = bench.code_sha256(*bench.KERNEL_SRCS)
    assert base != bench.code_sha256(bench.KERNEL_SRC)
    hdr = open(bench.KERNEL_SRCS[1], encoding="utf-8").read()
    p = tmp_path / "s.h"
    p.write_text(hdr.replace("if (j < nd) return j;", "if (j < nd) return nd - 1 - j;", 1), encoding="utf-8")
    assert bench.code_sha256(bench.KERNEL_SRC, str(p)) != base
    p.write_text("// comment\n" + hdr, encoding="utf-8")
    assert bench.code_sha256(bench.KERNEL_SRC, str(p)) == base
